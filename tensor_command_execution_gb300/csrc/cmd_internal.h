// cmd_internal.h - program encoding and launch parameters shared by the host
// lowering (cmd_api.cpp) and the CUDA executors (exec_*.cu). Not public.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#if defined(__CUDACC__)
#define CMDX_HD __host__ __device__
#else
#define CMDX_HD
#endif

namespace cmdx {

constexpr int kMaxRank = 4;
constexpr int kMaxLoads = 16;
constexpr int kMaxStores = 8;
constexpr int kMaxScalars = 16;
constexpr int kMaxSlots = 32;
constexpr int kMaxPrograms = 48;
constexpr int kMaxWords = 256;

// Executor families by register-slot count. The 2-, 4- and 8-slot tiers
// dispatch on one fused (opcode, dst, src) case; the wide tiers (16 and 32
// slots) fetch the source operand and then dispatch on (opcode, dst). (The
// 16-slot tier is numbered after the 32-slot one, which kept its number.)
enum Tier { kTier2 = 0, kTier4 = 1, kTier8 = 2, kTier32 = 3, kTier16 = 4 };
constexpr int kNumTiers = 5;
CMDX_HD constexpr int tier_slots(int tier) {
  return tier == kTier2 ? 2 : tier == kTier4 ? 4 : tier == kTier8 ? 8 : tier == kTier16 ? 16 : 32;
}
// The wide encoding (wd_word) and the two-level dispatch serve these tiers.
CMDX_HD constexpr bool tier_wide(int tier) { return tier == kTier16 || tier == kTier32; }
// Elements each thread keeps per slot in the contiguous executor: 16 in the
// 2-slot tier, 8 in the 4- and 8-slot tiers (16 in a second build of the
// base 4-slot tier, for programs whose loads are all 2-byte), 4 in the
// 16-slot tier and 2 in the 32-slot one. More elements per slot spread each
// program word's dispatch over more elements; fewer keep more CTAs
// resident. Measured for the 2-slot tier (A/B on one box, against 8 elements
// with the next chunk's loads prefetched in registers): bf16 add +8.7%,
// bf16 scale +17%, the 2^20-element fp32 add +16%, fp32 at 2^26-2^27
// within 1%; for its extended programs: packed-bit threshold +22%.
CMDX_HD constexpr int tier_vec(int tier, bool ext) {
  return tier == kTier2 ? 16 : tier == kTier32 ? 2 : tier == kTier16 ? 4 : 8;
}
// ... and in the generic executor, whose addressing needs more registers:
// 8, and 4 in the 8-slot tier.
CMDX_HD constexpr int tier_vec_strided(int tier) {
  return tier == kTier8 || tier == kTier16 ? 4 : tier == kTier32 ? 2 : 8;
}
// Resident 256-thread CTAs per SM each executor is compiled for (caps registers).
CMDX_HD constexpr int tier_min_blocks(int tier) { return tier_wide(tier) ? 2 : 3; }
// Program words a program may have: one less than its constant-memory row,
// so the interpreter's read-ahead of the word after the last stays in the row.
constexpr int kMaxProgramWords = kMaxWords - 1;

// Two-address binary ops: d = d (op) x, where x is a slot or a scalar.
// The R variants reverse the operands: d = x (op) d.
enum BinOp {
  kFAdd = 0, kFSub = 1, kFRsub = 2, kFMul = 3,
  kIAdd = 4, kISub = 5, kIRsub = 6, kIMul = 7,
  kFDiv = 8, kFRdiv = 9, kIDiv = 10, kIRdiv = 11,
  kFMin = 12, kFMax = 13, kIMin = 14, kIMax = 15,
  kNumBin = 16
};
// Unary ops: d = f(x).
enum UnOp { kFNeg = 0, kINeg = 1, kMov = 2, kFAbs = 3, kIAbs = 4, kI2F = 5, kF2I = 6, kNumUn = 7 };
// Comparisons: d = (d rel x) ? 1 : 0, floats (IEEE, ordered: false on NaN
// except NE), signed ints, unsigned ints. Swapping the operands maps LT <-> GT
// and LE <-> GE within each group (cmp_swap).
enum CmpOp {
  kCFLt = 0, kCFLe, kCFGt, kCFGe, kCFEq, kCFNe,
  kCILt = 6, kCILe, kCIGt, kCIGe, kCIEq, kCINe,
  kCULt = 12, kCULe, kCUGt, kCUGe,
  kNumCmp = 16
};
CMDX_HD constexpr int cmp_swap(int c) { return c % 6 < 2 ? c + 2 : c % 6 < 4 ? c - 2 : c; }
// Store element types, as numbered in cmd.h's cmd_dtype (B1: packed bits).
enum StoreType { kStF32 = 0, kStF16 = 1, kStBF16 = 2, kStI32 = 3, kStB1 = 4, kNumSt = 5 };

// ---- fused encoding (tiers 2, 4 and 8) ----------------------------------------
// word = case | aux << 16; aux is a scalar index (scalar ops) or an output
// index (stores). Case layout, for S slots (B = kNumBin, U = kNumUn,
// C = kNumCmp, T = kNumSt):
//   [0, B S^2)                binary op b, dst d, src slot s : b S^2 + d S + s
//   [B S^2, (B+U) S^2)        unary op u, dst d, src slot s  : B S^2 + u S^2 + d S + s
//   [(B+U) S^2, +B S)         binary op b with scalar src, dst d
//   then S cases              broadcast scalar into d
//   then T S cases            store slot s as type t
//   then                      end
//   then C S cases            compare c: d = d rel X (X = slot S - 1, the staging slot)
//   then C S cases            compare c: d = d rel scalar
//   then S^2 cases            select: d = X != 0 ? d : slot s
//   then S cases              select: d = X != 0 ? d : scalar
//   then 2 S cases            division o of d by a scalar through constants
//                             the host derives per launch (o = 0: binary32,
//                             scalars aux, aux + 1 = s, RN(1/s); o = 1:
//                             int32, scalars aux .. aux + 2 = d, magic, shift)
// Comparisons and selects read the staging slot X = S - 1, which the lowering
// fills right before (a program using it keeps slot S - 1 free), so that they
// take S cases each rather than S^2.
CMDX_HD constexpr uint32_t fz_bin(int S, int b, int d, int s) { return uint32_t(b * S * S + d * S + s); }
CMDX_HD constexpr uint32_t fz_un(int S, int u, int d, int s) { return uint32_t(kNumBin * S * S + u * S * S + d * S + s); }
CMDX_HD constexpr uint32_t fz_bin_scalar(int S, int b, int d) { return uint32_t((kNumBin + kNumUn) * S * S + b * S + d); }
CMDX_HD constexpr uint32_t fz_movs(int S, int d) { return uint32_t((kNumBin + kNumUn) * S * S + kNumBin * S + d); }
CMDX_HD constexpr uint32_t fz_store(int S, int t, int s) {
  return uint32_t((kNumBin + kNumUn) * S * S + (kNumBin + 1) * S + t * S + s);
}
CMDX_HD constexpr uint32_t fz_end(int S) {
  return uint32_t((kNumBin + kNumUn) * S * S + (kNumBin + 1 + kNumSt) * S);
}
CMDX_HD constexpr uint32_t fz_cmpx(int S, int c, int d) { return fz_end(S) + 1 + uint32_t(c * S + d); }
CMDX_HD constexpr uint32_t fz_cmps(int S, int c, int d) { return fz_end(S) + 1 + uint32_t((kNumCmp + c) * S + d); }
CMDX_HD constexpr uint32_t fz_sel(int S, int d, int s) { return fz_end(S) + 1 + uint32_t(2 * kNumCmp * S + d * S + s); }
CMDX_HD constexpr uint32_t fz_sels(int S, int d) { return fz_end(S) + 1 + uint32_t(2 * kNumCmp * S + S * S + d); }
CMDX_HD constexpr uint32_t fz_sdiv(int S, int o, int d) { return fz_sels(S, S) + uint32_t(o * S + d); }
CMDX_HD constexpr uint32_t fz_cases(int S) { return fz_sdiv(S, 2, 0); }  // number of cases

// Scalars the host derives at launch from a Load_Scalar value, for the
// divisions by a scalar (stored after the program's own scalars).
enum DerivedKind {
  kDerCopy = 0,     // the value itself
  kDerRecip = 1,    // binary32 RN(1 / s), or 0 when s is outside [2^-60, 2^60] (no fast path)
  kDerIMagic = 2,   // int32 division by d: the multiplier m - 2^32 (Granlund-Montgomery)
  kDerIShift = 3,   // ... the post-shift, with kSDivSlow set for d = 0 and d = -1
};
constexpr uint32_t kSDivSlow = 0x80000000u;

// ---- wide encoding (tiers 16 and 32) ---------------------------------------
// word = kind << 24 | d << 16 | s << 8 | aux. The source operand x is slot s,
// or scalar aux when the kind has kWScalar set. Selects read the staging
// slot X (the tier's last slot, 15 or 31) as their condition.
enum WideKind {
  kWBin0 = 0,    // + BinOp
  kWUn0 = 16,    // + UnOp
  kWStore0 = 23, // + StoreType, stores x to output aux
  kWEnd = 31,
  kWCmp0 = 32,   // + CmpOp: d = d rel x
  kWSel = 48,    // d = X != 0 ? d : x
  kWSDiv0 = 49,  // + o: d = d / scalars aux.. (the fused sdiv cases)
  kWScalar = 0x40
};
CMDX_HD constexpr uint32_t wd_word(int kind, int d, int s, int aux) {
  return uint32_t(kind) << 24 | uint32_t(d) << 16 | uint32_t(s) << 8 | uint32_t(aux);
}

// ---- launch parameters (passed by value as __grid_constant__) ---------------
// Bits of a kernel's device error word: a bounded wait that gave up.
constexpr uint32_t kErrConsumerWait = 1u << 0;  // data for a stage never arrived
constexpr uint32_t kErrProducerWait = 1u << 1;  // a stage was never freed
constexpr uint32_t kErrDrainWait = 1u << 2;     // copies still in flight at the stop never landed
constexpr uint32_t kErrDebugWait = 1u << 3;     // the test hook's wait (nothing completes it)

struct ContigParams {
  const void* in[kMaxLoads];
  void* out[kMaxStores];
  uint32_t scal[kMaxScalars];
  int64_t n;             // logical elements, a multiple of 32 * V
  uint32_t prog;         // program slot in constant memory
  uint32_t n_loads;
  uint8_t in_dt[kMaxLoads];
  // Row-contiguous launches (rows > 1): the elements are `rows` rows of
  // row_chunks warp chunks each (n = rows * row_chunks * 32 * V); row r of a
  // view starts r * ld elements after its base (ld = 0: one row read for
  // every row). One dense range otherwise (rows = 1, the ld unused).
  int32_t rows;
  int32_t row_chunks;
  int64_t in_ld[kMaxLoads];
  int64_t out_ld[kMaxStores];
  // Shifted launches (1-D, every tier but the 32-slot one): load j's first element
  // sits in_shift[j] elements past a vector boundary (0: aligned); every
  // store is aligned, and each view extends at least 4 elements before and
  // after the launch's range.
  uint8_t in_shift[kMaxLoads];
  uint8_t shifted;
};

// What the tile executor needs from the host. The logical index space is
// viewed as [b0][b1][row][col]: two tile dims (row, col) and up to two batch
// dims (size 1 when absent). Every store has unit stride along col; every
// load has unit stride along col ("row-direct") or along row ("transposed").
// The other tile dim of a load may have stride 0 (a broadcast row or column)
// and batch dims may have stride 0 (broadcast across the batch). The executor
// builds one TMA descriptor per load from this.
struct Tile2dLaunch {
  const void* in[kMaxLoads];
  int64_t in_ld[kMaxLoads];      // stride of the load's other tile dim (0 = broadcast)
  int64_t in_bst[kMaxLoads][2];  // batch strides (0 = broadcast)
  uint8_t in_dt[kMaxLoads];
  uint8_t in_trans[kMaxLoads];
  void* out[kMaxStores];
  int64_t out_ld[kMaxStores];     // row stride of each store
  int64_t out_bst[kMaxStores][2]; // batch strides of each store
  uint32_t scal[kMaxScalars];
  int64_t rows, cols;             // sizes of the two tile dims
  int64_t nb[2];                  // batch sizes (outer first)
  uint32_t prog;
  uint32_t n_loads;
  uint32_t* err;        // device error word of the kernel handle
  uint32_t debug;       // test hook: 1 = consumers wait on a barrier nobody arrives on
  uint64_t timeout_ns;  // limit of every device-side wait
};

// Bytes one pipeline stage of the tile executor holds for a load of element
// size es (a 64 x 64 box); the executor takes at most kTileStageLimit.
constexpr int tile_stage_bytes(int es) { return 64 * 64 * es; }
constexpr int kTileStageLimit = 48 * 1024;

// Unsigned division by an invariant divisor d >= 2 with a multiply-high:
// q = (t + ((n - t) >> 1)) >> (l - 1), t = mulhi64(m, n), l = ceil(log2 d),
// m = floor(2^64 (2^l - d) / d) + 1 (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, section 4).
struct FastDiv {
  uint64_t m;
  uint32_t l;   // 0 marks d == 1 (dimension skipped)
  uint32_t pad;
  int64_t d;
};

struct GenericParams {
  const void* in[kMaxLoads];
  void* out[kMaxStores];
  int64_t in_st[kMaxLoads][kMaxRank];   // strides, right-aligned to the merged rank
  int64_t out_st[kMaxStores][kMaxRank];
  FastDiv div[kMaxRank];                // merged sizes, right-aligned (leading dims = 1)
  uint32_t scal[kMaxScalars];
  int64_t n;
  uint32_t prog;
  uint32_t n_loads;
  uint32_t top;                         // outermost dim of size > 1 (kMaxRank - 1 if none)
  int64_t gap_at, gap;                  // logical index e >= gap_at stands for e + gap (1-D ranges)
  uint8_t in_dt[kMaxLoads];
};

// Host entry points of the executors. Each executor source is compiled once
// per tier and per op-set variant (CMDX_TIER, CMDX_EXT), so that the large
// per-tier interpreters compile in parallel and programs that use only the
// base ops (arithmetic, min/max, abs, conversions) run a loop that carries no
// code for the extended ones (division, comparisons, select, packed-bit
// stores); every such object keeps its own constant-memory program table.
// The functions below (exec_host.cpp) route a call to the object of a
// program's tier and variant.
#define CMDX_DECL_OBJ(t, v)                                                         \
  cudaError_t contig_upload_t##t##e##v(int slot, const uint32_t* words, int n);     \
  cudaError_t contig_launch_t##t##e##v(const ContigParams& p, cudaStream_t stream); \
  cudaError_t generic_upload_t##t##e##v(int slot, const uint32_t* words, int n);    \
  cudaError_t generic_launch_t##t##e##v(const GenericParams& p, cudaStream_t stream);
CMDX_DECL_OBJ(0, 0) CMDX_DECL_OBJ(1, 0) CMDX_DECL_OBJ(2, 0) CMDX_DECL_OBJ(3, 0) CMDX_DECL_OBJ(4, 0)
CMDX_DECL_OBJ(0, 1) CMDX_DECL_OBJ(1, 1) CMDX_DECL_OBJ(2, 1) CMDX_DECL_OBJ(3, 1) CMDX_DECL_OBJ(4, 1)
#undef CMDX_DECL_OBJ
// the extended 2-slot contiguous kernel built for four CTAs per SM
cudaError_t contig_upload_t0e1o4(int slot, const uint32_t* words, int n);
cudaError_t contig_launch_t0e1o4(const ContigParams& p, cudaStream_t stream);
// the base 4-slot contiguous kernel at 16 elements per slot (2-byte loads)
cudaError_t contig_upload_t1e0h16(int slot, const uint32_t* words, int n);
cudaError_t contig_launch_t1e0h16(const ContigParams& p, cudaStream_t stream);

// Write a compiled program into slot `slot` of every executor object of its
// tier and variant (ext: the program uses an extended op or store).
cudaError_t upload_program(int tier, bool ext, int slot, const uint32_t* words, int n);
// n must be a multiple of contig_chunk(tier, ext) elements.
// bits_only: every store of the program is packed bits (such programs read
// far more than they write, and the extended 2-slot tier runs them on its
// four-CTA build: measured, threshold_bits +12%, while one-word-per-element
// stores ran 1-6% slower there).
// half2: every load of the program is 2-byte (f16 or bf16); the base 4-slot
// tier then runs its 16-element build (its chunk is 512 elements).
cudaError_t contig_launch(int tier, bool ext, const ContigParams& p, cudaStream_t stream, bool bits_only = false,
                          bool half2 = false);
int contig_chunk(int tier, bool ext, bool half2 = false);
cudaError_t tile2d_launch(int tier, bool ext, const Tile2dLaunch& L, cudaStream_t stream);
cudaError_t generic_launch(int tier, bool ext, const GenericParams& p, cudaStream_t stream);

// Tile geometry of the tile2d executor.
constexpr int kTileRows = 64;
constexpr int kTileCols = 64;

}  // namespace cmdx
