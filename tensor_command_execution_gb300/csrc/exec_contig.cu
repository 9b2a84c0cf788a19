// exec_contig.cu - contiguous executor: every view is unit-stride and
// aligned for 4-element vectors, so each lane moves whole 16-byte (4-byte
// types) or 8-byte (2-byte types) vectors, a warp's access is contiguous, and
// the grid strides over warp-sized chunks of 32*V logical elements. It runs
// whole chunks only: the host hands a ragged tail (fewer than 32*V elements),
// and a head when every base is off the alignment by the same element count,
// to the generic executor, so the hot loop carries no bounds checks.
// Two more forms of the same kernel: a row walk over padded or sliced rows
// whose length is a whole number of chunks (ROWS), and shifted loads for
// views that sit off the stores' alignment by other element counts, read as
// aligned vectors and assembled from neighbouring lanes (SHIFT).
//
// Compiled once per tier and op-set variant: CMDX_TIER and CMDX_EXT select
// the kernel this object holds (and CMDX_OCC4 the four-CTA build of the
// extended 2-slot kernel, CMDX_HALF16 the 16-element build of the base
// 4-slot one).
#include "exec_common.cuh"

#if !defined(CMDX_TIER) || !defined(CMDX_EXT)
#error "exec_contig.cu is compiled per tier and variant, with -DCMDX_TIER=<0..4> -DCMDX_EXT=<0|1>"
#endif
#if CMDX_HALF16 && (CMDX_TIER != 1 || CMDX_EXT != 0)
#error "the 16-element build (CMDX_HALF16) is of the base 4-slot tier only"
#endif

namespace cmdx {

static __constant__ uint32_t c_prog[kMaxPrograms][kMaxWords];

// Elements per slot per thread of this object's kernel: the tier's, or 16
// in the CMDX_HALF16 build of the 4-slot tier (2-byte values carry half the
// bytes per element, so the interpreter's per-chunk cost is spread over
// twice the elements; measured, the bf16 chain Command +8%, while the fp32
// one loses 3% at 16).
CMDX_HD constexpr int contig_vec(int tier, bool ext) { return CMDX_HALF16 ? 16 : tier_vec(tier, ext); }

// Load one slot (V elements per lane) of a dense tensor of type dt. 2-byte
// types arrive packed, two to a word, in x[0 .. V/2); contig_widen expands
// them afterwards, so that every load of a chunk issues before any result is
// used (widening each group as it came would wait for its load before the
// next one issued).
template <int V>
__device__ __forceinline__ void contig_load(uint32_t (&x)[V], const void* base, int dt, int64_t e0) {
  using M = LaneMap<V>;
#pragma unroll
  for (int h = 0; h < M::NG; ++h) {
    const int64_t e = e0 + (int64_t)h * 32 * M::G;
    if (dt == 0 || dt == 3) {
      if constexpr (M::G == 4) {
        const uint4 q = ld_stream(reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(base) + e));
        x[4 * h] = q.x; x[4 * h + 1] = q.y; x[4 * h + 2] = q.z; x[4 * h + 3] = q.w;
      } else {
        const uint2 q = ld_stream(reinterpret_cast<const uint2*>(static_cast<const uint32_t*>(base) + e));
        x[2 * h] = q.x; x[2 * h + 1] = q.y;
      }
    } else {
      if constexpr (M::G == 4) {
        const uint2 q = ld_stream(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + e));
        x[2 * h] = q.x; x[2 * h + 1] = q.y;
      } else {
        x[h] = ld_stream(reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(base) + e));
      }
    }
  }
}

// Expand a 2-byte slot loaded by contig_load to one fp32 per register: word
// k holds elements 2k and 2k + 1 (from the last word down, so that no packed
// word is overwritten before it is read).
template <int V>
__device__ __forceinline__ void contig_widen(uint32_t (&x)[V], int dt) {
  if (dt == 1) {
#pragma unroll
    for (int k = V / 2 - 1; k >= 0; --k) {
      const uint32_t w = x[k];
      widen_f16x2(w, x[2 * k], x[2 * k + 1]);
    }
  } else if (dt == 2) {
#pragma unroll
    for (int k = V / 2 - 1; k >= 0; --k) {
      const uint32_t w = x[k];
      widen_bf16x2(w, x[2 * k], x[2 * k + 1]);
    }
  }
}

// A slot whose view starts r (1..3) elements past a vector boundary, while
// the launch's stores are aligned (x[1:] - x[:-1], say): each lane reads the
// aligned vectors that hold the start of its groups, from r elements before
// the view, in the same pattern as contig_load (its base is `a`, r elements
// before the view's); contig_shift then gives each lane its elements from
// its own vector and its right neighbour's. The last lane takes the next
// group's first vector, or for the chunk's last group one more vector, which
// it reads there (the host starts such a launch at least 4 elements into the
// views and leaves at least 4 after it, so these reads stay inside them).
// 2-byte values are still packed, two to a word; r is uniform over the launch.
template <int V>
__device__ __forceinline__ void contig_shift(uint32_t (&x)[V], const void* a, int dt, int r, int64_t e0, int lane) {
  using M = LaneMap<V>;
  static_assert(M::G == 4, "shifted loads take groups of 4 elements");
  const bool last = lane == 31;
  const bool r1 = r == 1, r2 = r == 2, hi = r >= 2;
  const uint32_t sh = (r & 1) * 16;
  // the vector after the chunk (read by the last lane only)
  const int64_t e_after = e0 + 4 + (int64_t)(M::NG - 1) * 32 * M::G;
  if (dt == 0 || dt == 3) {
    uint4 ex = make_uint4(0, 0, 0, 0);
    if (last) ex = ld_stream(reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(a) + e_after));
    const uint32_t exw[4] = {ex.x, ex.y, ex.z, ex.w};
#pragma unroll
    for (int h = 0; h < M::NG; ++h) {
      uint32_t n[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t dn = __shfl_down_sync(0xffffffffu, x[4 * h + q], 1);
        const uint32_t wrap = h + 1 < M::NG ? __shfl_sync(0xffffffffu, x[4 * (h + 1) + q], 0) : exw[q];
        n[q] = last ? wrap : dn;
      }
      // elements r .. r + 3 of (m0 m1 m2 m3 n0 n1 n2), selected without branching
      const uint32_t m1 = x[4 * h + 1], m2 = x[4 * h + 2], m3 = x[4 * h + 3];
      x[4 * h] = r1 ? m1 : r2 ? m2 : m3;
      x[4 * h + 1] = r1 ? m2 : r2 ? m3 : n[0];
      x[4 * h + 2] = r1 ? m3 : r2 ? n[0] : n[1];
      x[4 * h + 3] = r1 ? n[0] : r2 ? n[1] : n[2];
    }
  } else {
    uint2 ex = make_uint2(0, 0);
    if (last) ex = ld_stream(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a) + e_after));
    const uint32_t exw[2] = {ex.x, ex.y};
#pragma unroll
    for (int h = 0; h < M::NG; ++h) {
      uint32_t n[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t dn = __shfl_down_sync(0xffffffffu, x[2 * h + q], 1);
        const uint32_t wrap = h + 1 < M::NG ? __shfl_sync(0xffffffffu, x[2 * (h + 1) + q], 0) : exw[q];
        n[q] = last ? wrap : dn;
      }
      // elements r .. r + 3 (two to a word) of (m0 m1 n0 n1): words r / 2 ..
      // shifted right by 16 (r % 2) bits, without branching
      const uint32_t m0 = x[2 * h], m1 = x[2 * h + 1];
      const uint32_t w0 = hi ? m1 : m0, w1 = hi ? n[0] : m1, w2 = hi ? n[1] : n[0];
      x[2 * h] = __funnelshift_r(w0, w1, sh);
      x[2 * h + 1] = __funnelshift_r(w1, w2, sh);
    }
  }
}

// A view's row `row` (row-contiguous launches; row 0 is the base).
__device__ __forceinline__ const void* row_start(const void* base, int64_t row, int64_t ld, int dt) {
  return static_cast<const char*>(base) + row * ld * ((dt == 0 || dt == 3) ? 4 : 2);
}

template <int V, bool ROWS>
struct ContigStore {
  const ContigParams& p;
  int64_t e0;
  int64_t row;  // (row-contiguous launches)

  template <int T>
  __device__ __forceinline__ void store(const uint32_t (&x)[V], uint32_t o) const {
    using M = LaneMap<V>;
    void* base = p.out[o];
    if constexpr (ROWS && T != kStB1)  // (packed-bit stores never take rows)
      base = static_cast<char*>(base) + row * p.out_ld[o] * ((T == kStF32 || T == kStI32) ? 4 : 2);
    if constexpr (T == kStB1) {
      // one bit per element (min(x, 1) is 1 exactly when x != 0)
      constexpr int G = M::G, L = 32 / G;
      const int lane = threadIdx.x & 31;
      const int64_t chunk = e0 - (int64_t)lane * G;  // a multiple of 32 * V
      if constexpr (G == 4 && M::NG == 4) {
        // The lane's 16 bits, element 4h + j at bit 4h + j. The 32 elements
        // of word h of an 8-lane group are nibble h of its lanes: two
        // xor-butterflies exchange the lane index bits 0 and 1 with the
        // nibble index bits, and one shuffle then gives lane 2h + k of the
        // group bits 16k .. 16k + 15 of its word h, stored as a halfword (a
        // warp writes its 64 bytes with one store).
        uint32_t v = min(x[0], 1u);
#pragma unroll
        for (int k = 1; k < 16; ++k) v += min(x[k], 1u) << k;
        const bool b0 = lane & 1, b1 = lane & 2;
        const uint32_t k0 = b0 ? 0xF0F0u : 0x0F0Fu, k1 = b1 ? 0xFF00u : 0x00FFu;
        uint32_t t = __shfl_xor_sync(0xffffffffu, v, 1) & k0;
        v = (v & k0) | __funnelshift_r(t, t, b0 ? 4 : 28);
        t = __shfl_xor_sync(0xffffffffu, v, 2) & k1;
        v = (v & k1) | __funnelshift_r(t, t, b1 ? 8 : 24);
        const int q = lane & 7;
        v = __shfl_sync(0xffffffffu, v, (lane & ~7) | ((q & 1) << 2) | (q >> 1));
        st_stream(reinterpret_cast<uint16_t*>(static_cast<uint32_t*>(base) + chunk / 32) + 8 * (q >> 1) +
                      2 * (lane >> 3) + (q & 1),
                  (uint16_t)v);
      } else {
        // a lane's G bits of group h go to bits G * (lane % L) .. of word
        // (group start) / 32 + lane / L, L = 32 / G lanes sharing a word; an
        // xor-shuffle tree ORs them together
#pragma unroll
        for (int h = 0; h < M::NG; ++h) {
          uint32_t bits = min(x[h * G], 1u);
#pragma unroll
          for (int j = 1; j < G; ++j) bits += min(x[h * G + j], 1u) << j;
          bits <<= G * (lane % L);
#pragma unroll
          for (int m = 1; m < L; m <<= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, m);
          if (lane % L == 0)
            st_stream(static_cast<uint32_t*>(base) + (chunk + (int64_t)h * 32 * G) / 32 + lane / L, bits);
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < M::NG; ++h) {
        const int64_t e = e0 + (int64_t)h * 32 * M::G;
        const uint32_t* v = &x[h * M::G];
        if constexpr (T == kStF32 || T == kStI32) {
          if constexpr (M::G == 4)
            st_stream(reinterpret_cast<uint4*>(static_cast<uint32_t*>(base) + e), make_uint4(v[0], v[1], v[2], v[3]));
          else
            st_stream(reinterpret_cast<uint2*>(static_cast<uint32_t*>(base) + e), make_uint2(v[0], v[1]));
        } else {
          auto nar = [](uint32_t a, uint32_t b) {
            if constexpr (T == kStF16) return narrow_f16x2(a, b);
            else return narrow_bf16x2(a, b);
          };
          if constexpr (M::G == 4)
            st_stream(reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + e),
                      make_uint2(nar(v[0], v[1]), nar(v[2], v[3])));
          else
            st_stream(reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(base) + e), nar(v[0], v[1]));
        }
      }
    }
  }
};

// One warp chunk: elements e0 .. of each view (of its row `row` when ROWS;
// with loads off the stores' alignment when SHIFT).
template <int TIER, bool EXT, bool ROWS, bool SHIFT>
__device__ __forceinline__ void contig_run_chunk(const ContigParams& p, const uint32_t* prog, int64_t e0,
                                                 int64_t row) {
  constexpr int S = tier_slots(TIER);
  constexpr int V = contig_vec(TIER, EXT);
  constexpr int NL = S < kMaxLoads ? S : kMaxLoads;
  uint32_t r[S][V];
  // (a shifted load reads from the aligned vector before its first element)
  auto base_of = [&](int j) -> const void* {
    const void* b = p.in[j];
    if constexpr (ROWS) b = row_start(b, row, p.in_ld[j], p.in_dt[j]);
    if constexpr (SHIFT) b = static_cast<const char*>(b) - (int)p.in_shift[j] * ((p.in_dt[j] == 0 || p.in_dt[j] == 3) ? 4 : 2);
    return b;
  };
#pragma unroll
  for (int j = 0; j < NL; ++j)
    if (j < (int)p.n_loads) contig_load<V>(r[j], base_of(j), p.in_dt[j], e0);
  if constexpr (SHIFT) {
#pragma unroll
    for (int j = 0; j < NL; ++j)
      if (j < (int)p.n_loads && p.in_shift[j])
        contig_shift<V>(r[j], base_of(j), p.in_dt[j], p.in_shift[j], e0, threadIdx.x & 31);
  }
#pragma unroll
  for (int j = 0; j < NL; ++j)
    if (j < (int)p.n_loads) contig_widen<V>(r[j], p.in_dt[j]);
  ContigStore<V, ROWS> st{p, e0, row};
  run_program<TIER, V, EXT>(r, prog, p.scal, st);
}

// MINB: resident CTAs per SM the registers are sized for (one object of the
// extended 2-slot tier is built for 4 instead of 3, for packed-bit programs).
// ROWS: a row-contiguous launch; warp w takes chunk w % row_chunks of row
// w / row_chunks, the pair stepped by the grid's warp count with a carry
// instead of dividing per chunk.
template <int TIER, bool EXT, int MINB, bool ROWS, bool SHIFT>
__global__ void __launch_bounds__(256, MINB) contig_kernel(const __grid_constant__ ContigParams p) {
  constexpr int V = contig_vec(TIER, EXT);
  using M = LaneMap<V>;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t* prog = c_prog[p.prog];
  int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if constexpr (!EXT) {
    // A launch of at most one chunk per warp (a small one) cannot pipeline
    // its loads, so it would take the DRAM latency after the wait for the
    // previous launch. Its warps ask L2 for their chunk of every load
    // first: a prefetch returns nothing to the thread, and L2 is where
    // every SM's accesses meet, so a line that the previous launch writes
    // afterwards is updated there and never read stale.
    const int64_t n_chunks = ROWS ? (int64_t)p.rows * p.row_chunks : p.n / M::W;
    if (n_chunks <= nwarps && w < n_chunks) {
      int64_t e_first = w * M::W, row0 = 0;
      if constexpr (ROWS) {
        row0 = w / p.row_chunks;
        e_first = (w - row0 * p.row_chunks) * M::W;
      }
      e_first += (int64_t)lane * M::G;
      constexpr int NL = tier_slots(TIER) < kMaxLoads ? tier_slots(TIER) : kMaxLoads;
#pragma unroll
      for (int j = 0; j < NL; ++j)
        if (j < (int)p.n_loads) {
          const void* b = p.in[j];
          if constexpr (ROWS) b = row_start(b, row0, p.in_ld[j], p.in_dt[j]);
          const int es = (p.in_dt[j] == 0 || p.in_dt[j] == 3) ? 4 : 2;
#pragma unroll
          for (int h = 0; h < M::NG; ++h)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(b) +
                                                          (e_first + (int64_t)h * 32 * M::G) * es));
        }
    }
  }
  pdl_wait();
  pdl_trigger();
  if constexpr (!ROWS) {
    const int64_t n_chunks = p.n / M::W;  // the host passes a multiple of W
    for (; w < n_chunks; w += nwarps)
      contig_run_chunk<TIER, EXT, false, SHIFT>(p, prog, w * M::W + (int64_t)lane * M::G, 0);
  } else {
    // rows and row_chunks are below 2^31, and so is the grid's warp count
    const int rc = p.row_chunks;
    int row = (int)(w / rc), c = (int)(w % rc);
    const int drow = (int)(nwarps / rc), dc = (int)(nwarps % rc);
    while (row < p.rows) {
      contig_run_chunk<TIER, EXT, true, SHIFT>(p, prog, (int64_t)c * M::W + (int64_t)lane * M::G, row);
      c += dc;
      row += drow;
      if (c >= rc) {
        c -= rc;
        ++row;
      }
    }
  }
}

cudaError_t CMDX_TIER_NAME(contig_upload_t)(int slot, const uint32_t* words, int n) {
  return cudaMemcpyToSymbol(c_prog, words, sizeof(uint32_t) * n, sizeof(uint32_t) * kMaxWords * slot);
}

template <int TIER, bool EXT, bool ROWS, bool SHIFT = false>
static cudaError_t launch_tier(const ContigParams& p, cudaStream_t stream) {
  // (the 2-slot tier's dense-range kernel fits 64 registers and so runs four
  // CTAs per SM; its row-walking one is held to the same)
  // (the 8-slot kernel with shifted loads is held to two CTAs per SM: at
  // three it spilled 160 bytes)
  constexpr int MINB = (CMDX_OCC4 || (ROWS && !SHIFT && TIER == kTier2 && !EXT)) ? 4
                       : (SHIFT && TIER == kTier8)                     ? 2
                                                                       : tier_min_blocks(TIER);
  constexpr int V = contig_vec(TIER, EXT);
  constexpr int kBlock = 256;
  static DeviceCache grid_cache;  // (static storage: zero before first use)
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t work_blocks = (p.n + (int64_t)kBlock * V - 1) / ((int64_t)kBlock * V);
  int full_grid = grid_cache.get(dev);
  if (full_grid == 0) {
    full_grid = persistent_grid(contig_kernel<TIER, EXT, MINB, ROWS, SHIFT>, kBlock, 0, INT64_MAX);
    grid_cache.put(dev, full_grid);
  }
  const int grid = (int)(work_blocks < full_grid ? work_blocks : full_grid);
  return launch_pdl(contig_kernel<TIER, EXT, MINB, ROWS, SHIFT>, grid, kBlock, 0, stream, p);
}

// The extended 8-slot interpreter is the largest: each more form of its
// kernel adds about half a minute to its object's compile, the build's
// longest, so that object holds the dense-range kernel alone (the host
// sends it no row walk and no shifted launch; such views take the tile or
// generic executor).
constexpr bool kDenseOnly = CMDX_TIER == kTier8 && CMDX_EXT;
// Objects whose kernels take shifted loads: every tier whose lanes hold
// groups of 4 elements (not the 32-slot one), not the 16-element or
// four-CTA builds (the host never sends them shifted launches).
constexpr bool kShiftObject = CMDX_TIER != kTier32 && !kDenseOnly && !CMDX_HALF16 && !CMDX_OCC4;

cudaError_t CMDX_TIER_NAME(contig_launch_t)(const ContigParams& p, cudaStream_t stream) {
  if (p.shifted) {
    if constexpr (kShiftObject) {
      if (p.rows > 1) return launch_tier<CMDX_TIER, CMDX_EXT != 0, true, true>(p, stream);
      return launch_tier<CMDX_TIER, CMDX_EXT != 0, false, true>(p, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (p.rows > 1) {
    if constexpr (!kDenseOnly) return launch_tier<CMDX_TIER, CMDX_EXT != 0, true>(p, stream);
    return cudaErrorInvalidValue;
  }
  return launch_tier<CMDX_TIER, CMDX_EXT != 0, false>(p, stream);
}

}  // namespace cmdx
