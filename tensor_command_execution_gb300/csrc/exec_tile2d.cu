// exec_tile2d.cu - 2-D strided executor: views that are row-direct (element
// (i, j) at i*ld + j) or transposed (element (i, j) at i + j*ld), stores
// row-direct.
//
// The logical index space is cut into 64 x 64 tiles that persistent CTAs walk
// in a grid stride. One producer warp stages every load of a tile into shared
// memory with TMA (cp.async.bulk.tensor.2d, 128-byte swizzle, no multicast),
// through a ring of pipeline stages guarded by mbarriers: "full" completes
// when a stage's bytes have landed, "empty" when all consumer warps have read
// it. Eight consumer warps read the stage, run the program and store straight
// to global memory with 16-byte vector stores. A transposed view arrives in
// its physical layout (one box row per logical column) and is read across box
// rows; each lane walks them in an order of its own (step k, box row k ^ cj
// of its group) so that the eight lanes of a tile row hit distinct banks,
// then permutes its registers back.
//
// Every wait on an mbarrier is bounded by a time limit; a wait that runs out
// records a code in the kernel's device error word and the CTA stops (after
// waiting, again bounded, for the copies it issued), so a stuck copy cannot
// hang the GPU. cmd_sync_status reports it.
//
// rocRoller, "Design Overview", section "Kernel Graph": the coordinate
// transforms map each logical index to a tensor offset through sizes and
// strides; tiling and staging through shared memory is how this executor
// makes those transforms coalesce (the pages' own generator stages tiles
// through LDS on AMD hardware).
//
// Compiled once per tier (CMDX_TIER 0..2), view variant (CMDX_ND 0: plain
// 2-D views; 1: batch dims, broadcast loads or descriptors of another rank)
// and op-set variant (CMDX_EXT): each object holds one kernel. The TMA
// descriptors are encoded on the host (exec_host.cpp).
#include "exec_common.cuh"
#include "exec_pipe.cuh"
#include "exec_tile2d.h"

#if !defined(CMDX_TIER) || !defined(CMDX_ND) || !defined(CMDX_EXT)
#error "exec_tile2d.cu is compiled per variant, with -DCMDX_TIER=<0..2> -DCMDX_ND=<0|1> -DCMDX_EXT=<0|1>"
#endif
// tile2d_<f>_t<tier>n<nd>e<ext>: this object's entry points
#define CMDX_TILE_NAME(f) \
  CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(f, CMDX_TIER), n), CMDX_ND), e), CMDX_EXT)

namespace cmdx {

static __constant__ uint32_t c_prog[kMaxPrograms][kMaxWords];

// One box of a descriptor of rank 1..5 at coordinates c[0..rank).
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int rank, const int32_t (&c)[5],
                                         uint32_t bar) {
  const uint64_t m = reinterpret_cast<uint64_t>(map);
  switch (rank) {
    case 1:
      asm volatile(
          "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];"
          ::"r"(dst), "l"(m), "r"(c[0]), "r"(bar) : "memory");
      break;
    case 2:
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
          ::"r"(dst), "l"(m), "r"(c[0]), "r"(c[1]), "r"(bar) : "memory");
      break;
    case 3:
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
          ::"r"(dst), "l"(m), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(bar) : "memory");
      break;
    case 4:
      asm volatile(
          "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
          "[%6];"
          ::"r"(dst), "l"(m), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(bar) : "memory");
      break;
    default:
      asm volatile(
          "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], "
          "[%7];"
          ::"r"(dst), "l"(m), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(bar) : "memory");
      break;
  }
}

// ---- reading a stage -----------------------------------------------------------
// A 64 x 64 box with 128-byte rows and the 128-byte swizzle keeps 16-byte
// chunk c of row q at q*128 + ((c ^ (q % 8)) * 16); 4-byte views use two boxes
// of 32 elements per row, the second 8 KB after the first.
__device__ __forceinline__ void xor_perm8(uint32_t (&y)[8], int c);

// Transposed reads: logical (li, 8 cj + m) is element li of box row
// q = 8 cj + m. Step k of a lane reads m = k ^ cj, so the lanes of a tile row
// (cj = 0..7) see eight different q % 8 and, under the swizzle, eight
// different chunks. Its address is then one per-thread base XOR k * 0x90:
// bits 7..9 (q % 8 = k ^ cj) and bits 4..6 (the chunk, (li / 8) ^ k ^ cj)
// both flip with k, and the base's own bits 4..9 start at cj and li / 8 ^ cj.
__device__ __forceinline__ uint32_t trans_base(uint32_t stage, bool half, int li, int cj) {
  const uint32_t c = (uint32_t)cj;
  if (half) {
    const uint32_t ch = (uint32_t)li >> 3;
    return (stage + c * 1024 + (li & 7) * 2) | (c << 7) | ((ch ^ c) << 4);
  }
  const uint32_t lr = li & 31;
  return (stage + (li >> 5) * kBoxBytes + c * 1024 + (lr & 3) * 4) | (c << 7) | (((lr >> 2) ^ c) << 4);
}

// Row-direct: logical (li, 8 cj .. 8 cj + 7).
__device__ __forceinline__ void read_row(uint32_t (&x)[8], uint32_t stage, int dt, int li, int cj) {
  const uint32_t sw = li & 7;
  if (dt == 1 || dt == 2) {
    const uint4 a = lds128(stage + li * 128 + ((cj ^ sw) << 4));
    if (dt == 1) {
      widen_f16x2(a.x, x[0], x[1]); widen_f16x2(a.y, x[2], x[3]);
      widen_f16x2(a.z, x[4], x[5]); widen_f16x2(a.w, x[6], x[7]);
    } else {
      widen_bf16x2(a.x, x[0], x[1]); widen_bf16x2(a.y, x[2], x[3]);
      widen_bf16x2(a.z, x[4], x[5]); widen_bf16x2(a.w, x[6], x[7]);
    }
  } else {
    // columns 8 cj.. live in box cj / 4, chunks 2 (cj % 4) and 2 (cj % 4) + 1;
    // lanes of the second box take their chunks in the other order so a
    // tile row's eight lanes cover all eight chunk positions at each access
    const uint32_t box = stage + (cj >> 2) * kBoxBytes + li * 128;
    const uint32_t c0 = (cj & 3) * 2;
    const bool flip = (cj >> 2) & 1;
    const uint4 a = lds128(box + (((c0 + (flip ? 1 : 0)) ^ sw) << 4));
    const uint4 b = lds128(box + (((c0 + (flip ? 0 : 1)) ^ sw) << 4));
    const uint4 lo = flip ? b : a, hi = flip ? a : b;
    x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
    x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
  }
}

// Transposed, one row: x[m] = logical (li, 8 cj + m).
__device__ __forceinline__ void read_trans(uint32_t (&x)[8], uint32_t stage, int dt, int li, int cj) {
  uint32_t y[8];
  const bool half = dt == 1 || dt == 2;
  const uint32_t a = trans_base(stage, half, li, cj);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (half) {
      const uint32_t h = lds16(a ^ (uint32_t)(k * 0x90));
      y[k] = dt == 1 ? widen_f16((uint16_t)h) : widen_bf16((uint16_t)h);
    } else {
      y[k] = lds32(a ^ (uint32_t)(k * 0x90));
    }
  }
  xor_perm8(y, cj);
#pragma unroll
  for (int m = 0; m < 8; ++m) x[m] = y[m];
}


// y[m] = y[m ^ c] for a thread-constant c: conditional swaps of the pairs
// that differ in bit 1, 2 and 4 of the index.
__device__ __forceinline__ void xor_perm8(uint32_t (&y)[8], int c) {
#pragma unroll
  for (int b = 1; b < 8; b <<= 1) {
    const bool f = (c & b) != 0;
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if ((m & b) == 0) {
        const uint32_t u = y[m], v = y[m | b];
        y[m] = f ? v : u;
        y[m | b] = f ? u : v;
      }
  }
}

// Two rows per thread: x[0..7] is box row la, x[8..15] box row lb.
__device__ __forceinline__ void read_row2(uint32_t (&x)[16], uint32_t stage, int dt, int la, int lb, int cj) {
  uint32_t a[8], b[8];
  read_row(a, stage, dt, la, cj);
  read_row(b, stage, dt, lb, cj);
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    x[m] = a[m];
    x[8 + m] = b[m];
  }
}

// Transposed, two rows: rows li and li + 1 of box row q are adjacent, so one
// 32-bit (2-byte types) or 64-bit (4-byte types) load fetches both.
__device__ __forceinline__ void read_trans2(uint32_t (&x)[16], uint32_t stage, int dt, int li, int cj) {
  uint32_t y0[8], y1[8];
  const bool half = dt == 1 || dt == 2;
  const uint32_t a = trans_base(stage, half, li, cj);
  if (half) {
#pragma unroll
    for (int k = 0; k < 8; ++k) y0[k] = lds32(a ^ (uint32_t)(k * 0x90));
    xor_perm8(y0, cj);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (dt == 1) {
        widen_f16x2(y0[m], x[m], x[8 + m]);
      } else {
        widen_bf16x2(y0[m], x[m], x[8 + m]);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint2 v = lds64(a ^ (uint32_t)(k * 0x90));
      y0[k] = v.x;
      y1[k] = v.y;
    }
    xor_perm8(y0, cj);
    xor_perm8(y1, cj);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      x[m] = y0[m];
      x[8 + m] = y1[m];
    }
  }
}

// Transposed, split layout (batched launches of the 2-slot tier, 4-byte
// loads): the host split the load's column dim into (column / 8, column % 8),
// the group first, so logical (li, 8 cj + k) is box row cj + 8 k. Under the
// 128-byte swizzle (chunk ^= box row % 8 = cj) a tile row's eight lanes read
// eight distinct chunks at every step, and step k of a lane is register k:
// eight loads at fixed offsets from one address, with no permutation after.
__device__ __forceinline__ uint32_t split_base(uint32_t stage, bool half, int li, int cj) {
  if (half) return stage + cj * 128 + ((((uint32_t)li >> 3) ^ (uint32_t)cj) << 4) + (li & 7) * 2;
  const uint32_t lr = li & 31;
  return stage + (li >> 5) * kBoxBytes + cj * 128 + (((lr >> 2) ^ (uint32_t)cj) << 4) + (lr & 3) * 4;
}

// Rows li and li + 1: one 32-bit (2-byte types) or 64-bit load per step.
__device__ __forceinline__ void read_trans2_split(uint32_t (&x)[16], uint32_t stage, int dt, int li, int cj) {
  const bool half = dt == 1 || dt == 2;
  const uint32_t a = split_base(stage, half, li, cj);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (half) {
      const uint32_t v = lds32(a + k * 1024);
      if (dt == 1) widen_f16x2(v, x[k], x[8 + k]);
      else widen_bf16x2(v, x[k], x[8 + k]);
    } else {
      const uint2 v = lds64(a + k * 1024);
      x[k] = v.x;
      x[8 + k] = v.y;
    }
  }
}

// A broadcast column (transposed load whose column stride is 0): the box has
// one row, element li of it is the value of every column of row li.
__device__ __forceinline__ uint32_t read_bcast_col(uint32_t stage, int dt, int li) {
  if (dt == 1 || dt == 2) {
    const uint32_t h = lds16(stage + ((((uint32_t)li >> 3) ^ 0u) << 4) + (li & 7) * 2);
    return dt == 1 ? widen_f16((uint16_t)h) : widen_bf16((uint16_t)h);
  }
  return lds32(stage + (li >> 5) * kBoxBytes + ((((uint32_t)li & 31) >> 2) << 4) + (li & 3) * 4);
}

// The tiles a CTA visits, t = blockIdx.x, + gridDim.x, ..., as the digits of
// t = ((b0 * nb1 + b1) * tiles_r + tr) * tiles_c + tc, advanced by adding
// the digits of gridDim.x with carries: no division per tile (used by the
// producer of batched launches; measured, it did not pay elsewhere).
struct TileWalk {
  uint32_t tc, tr, b1, b0;   // digits of t (tr holds t / tiles_c when !nd)
  uint32_t dc, dr, d1, d0;   // digits of the stride
  __device__ __forceinline__ void init(const Tile2dParams& p, bool nd, uint32_t t, uint32_t g) {
    tc = t % p.tiles_c;
    dc = g % p.tiles_c;
    uint32_t t1 = t / p.tiles_c, g1 = g / p.tiles_c;
    if (nd) {
      tr = t1 % p.tiles_r;
      dr = g1 % p.tiles_r;
      const uint32_t t2 = t1 / p.tiles_r, g2 = g1 / p.tiles_r;
      b1 = t2 % p.nb1;
      b0 = t2 / p.nb1;
      d1 = g2 % p.nb1;
      d0 = g2 / p.nb1;
    } else {
      tr = t1;
      dr = g1;
      b1 = b0 = d1 = d0 = 0;
    }
  }
  __device__ __forceinline__ void next(const Tile2dParams& p, bool nd) {
    tc += dc;
    uint32_t c = tc >= p.tiles_c;
    if (c) tc -= p.tiles_c;
    tr += dr + c;
    if (nd) {
      c = tr >= p.tiles_r;
      if (c) tr -= p.tiles_r;
      b1 += d1 + c;
      c = b1 >= p.nb1;
      if (c) b1 -= p.nb1;
      b0 += d0 + c;
    }
  }
};

template <bool ND>
struct TileStore {
  const Tile2dParams& p;
  int64_t i, j;
  bool full;
  int ncols_left;
  uint32_t b0, b1;

  template <int T>
  __device__ __forceinline__ void store(const uint32_t (&x)[8], uint32_t o) const {
    // packed-bit stores never come here: the host plans programs that have
    // them onto the contiguous or generic executor
    if constexpr (T == kStB1) return;
    void* base = p.out[o];
    int64_t off = i * p.out_ld[o] + j;
    if (ND) off += (int64_t)b0 * p.out_bst[o][0] + (int64_t)b1 * p.out_bst[o][1];
    if (full) {
      if constexpr (T == kStF32 || T == kStI32) {
        uint4* q = reinterpret_cast<uint4*>(static_cast<uint32_t*>(base) + off);
        st_stream(q, make_uint4(x[0], x[1], x[2], x[3]));
        st_stream(q + 1, make_uint4(x[4], x[5], x[6], x[7]));
      } else if constexpr (T == kStF16) {
        st_stream(reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + off),
                  make_uint4(narrow_f16x2(x[0], x[1]), narrow_f16x2(x[2], x[3]), narrow_f16x2(x[4], x[5]),
                             narrow_f16x2(x[6], x[7])));
      } else {
        st_stream(reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + off),
                  make_uint4(narrow_bf16x2(x[0], x[1]), narrow_bf16x2(x[2], x[3]), narrow_bf16x2(x[4], x[5]),
                             narrow_bf16x2(x[6], x[7])));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < ncols_left) st_elem<T>(base, off + k, x[k]);
    }
  }
};

// Two rows per thread: x[0..7] to row i, x[8..15] to row i + 1 (if it
// exists); the second row's state is derived from the first when it is
// stored (the consumers are short of registers).
template <bool ND>
struct TileStore2 {
  TileStore<ND> lo;
  bool second;

  template <int T>
  __device__ __forceinline__ void store(const uint32_t (&x)[16], uint32_t o) const {
    uint32_t a[8], b[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      a[m] = x[m];
      b[m] = x[8 + m];
    }
    lo.template store<T>(a, o);
    if (second) {
      TileStore<ND> hi = lo;
      hi.i += 1;
      hi.template store<T>(b, o);
    }
  }
};

// Stage index and phase parity of a pipeline ring of ns stages, stepped once
// per tile (no division per tile).
struct StageRing {
  uint32_t s = 0, ph = 0;
  __device__ __forceinline__ void next(uint32_t ns) {
    if (++s == ns) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// The producer lane of a tile CTA: for each tile of the CTA's grid stride,
// wait for its stage to be free, publish the tile's coordinates beside the
// stage's barrier and issue every load's TMA boxes into the stage. A wait
// that runs out records a code in the error word; the lane then waits
// (bounded) for the copies it issued and returns.
template <bool ND>
__device__ __forceinline__ void tile_produce(const Tile2dParams& p, uint32_t full_bar, uint32_t empty_bar,
                                             uint32_t coords, uint32_t stages, uint32_t ns) {
  uint32_t n = 0;
  bool ok = true;
  TileWalk tw;  // (batched launches: it replaces three divisions a tile)
  if (ND) tw.init(p, true, blockIdx.x, gridDim.x);
  StageRing ring;
  for (uint32_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++n, ring.next(ns)) {
    const uint32_t s = ring.s, ph = ring.ph;
    if (!mbar_wait(empty_bar + 8 * s, ph ^ 1, p.timeout_ns)) {
      atomicOr(p.err, kErrProducerWait);
      ok = false;
      break;
    }
    // t = ((b0 * nb1 + b1) * tiles_r + tile row) * tiles_c + tile column
    uint32_t tc, tr;
    int32_t bc1 = 0, bc2 = 0;  // batch coordinates b0, b1
    if (ND) {
      tc = tw.tc;
      tr = tw.tr;
      bc1 = (int32_t)tw.b0;
      bc2 = (int32_t)tw.b1;
      tw.next(p, true);
    } else {
      // tiles in groups of group_rows tile rows, column by column within a
      // group: the tiles in flight at once then cover a block of tile rows
      // and columns, so a transposed operand is read in runs of
      // 128 B x group_rows from each of its rows, not 128 B
      const uint32_t per_group = p.group_rows * p.tiles_c;
      const uint32_t g = t / per_group, rem = t - g * per_group;
      const uint32_t g0 = g * p.group_rows;
      const uint32_t h = p.tiles_r - g0 < p.group_rows ? p.tiles_r - g0 : p.group_rows;
      tc = rem / h;
      tr = g0 + (rem - tc * h);
    }
    const int32_t i0 = (int32_t)(tr * kTileRows), j0 = (int32_t)(tc * kTileCols);
    const uint32_t fb = full_bar + 8 * s;
    // the tile's coordinates for the consumers (published by the arrive
    // below, whose release orders this store before the phase completes)
    sts128(coords + 16 * s, make_uint4(tr, tc, (uint32_t)bc1, (uint32_t)bc2));
    mbar_arrive_expect_tx(fb, p.tx_bytes);
    const uint32_t st = stages + s * p.stage_bytes;
    for (uint32_t j = 0; j < p.n_loads; ++j) {
      const uint32_t dst = st + p.load_off[j];
      const bool wide = !(p.in_dt[j] == 1 || p.in_dt[j] == 2);
      // dim 0 runs along the load's unit-stride tile dim; dims 1.. take the
      // other tile coordinate or a batch coordinate, as routed on the host
      const int32_t inner = p.in_trans[j] ? i0 : j0, outer = p.in_trans[j] ? j0 : i0;
      int32_t c[5] = {inner, outer, 0, 0, 0};
      if (ND) {
        // descriptor dims 1..: the other tile dim (src 0), a batch dim
        // (1, 2), or the two halves of a split column dim (3: column / 8,
        // 4: column % 8, whose box always starts at 0)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t src = p.in_src[j][k];
          c[k + 1] = src == 0 ? outer : src == 1 ? bc1 : src == 2 ? bc2 : src == 3 ? outer / 8 : 0;
        }
      }
      const int rank = ND ? p.in_rank[j] : 2;
      tma_load(dst, &p.maps[j], rank, c, fb);
      if (wide) {
        c[0] = inner + 32;
        tma_load(dst + kBoxBytes, &p.maps[j], rank, c, fb);
      }
    }
  }
  if (!ok) {
    // wait (bounded) for the copies still in flight into this CTA's stages
    const uint32_t pend = n < ns ? n : ns;
    for (uint32_t q = n - pend; q < n; ++q)
      if (!mbar_wait(full_bar + 8 * (q % ns), (q / ns) & 1, p.timeout_ns)) atomicOr(p.err, kErrDrainWait);
  }
}

// Resident CTAs per SM the register budget is sized for (the 2-slot tier
// fits four in 56 registers; shared memory then allows 3 stages of 16 KB).
CMDX_HD constexpr int tile_min_blocks(int tier) { return tier == kTier2 ? 4 : 2; }
// Rows each consumer thread handles per tile pass: 2 in the 2- and 4-slot tiers.
CMDX_HD constexpr int tile_rows_per_thread(int tier) { return tier == kTier8 ? 1 : 2; }

// ND: the launch has batch dims or broadcast loads. Plain 2-D launches
// compile without that bookkeeping (the consumer warps are issue-bound).
template <int TIER, bool ND, bool EXT>
__global__ void __launch_bounds__(kThreads, tile_min_blocks(TIER)) tile2d_kernel(const __grid_constant__ Tile2dParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int S = tier_slots(TIER);
  constexpr int NL = S < kMaxLoads ? S : kMaxLoads;
  const uint32_t base = smem_u32(smem);
  const uint32_t full_bar = base;                    // kMaxStages x 8 bytes
  const uint32_t empty_bar = base + 8 * kMaxStages;  // kMaxStages x 8 bytes
  const uint32_t debug_bar = base + 16 * kMaxStages;
  const uint32_t coords = base + 32 * kMaxStages;    // kMaxStages x 16 bytes: the stage's tile
  const uint32_t stages = base + kBarrierBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ns = p.n_stages;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < ns; ++s) {
      mbar_init(full_bar + 8 * s, 1);
      mbar_init(empty_bar + 8 * s, kConsumerWarps);
    }
    mbar_init(debug_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // (barrier setup above touches only shared memory; every global access,
  // the producer's TMA loads included, comes after the previous kernel)
  pdl_wait();
  pdl_trigger();

  if (warp == kConsumerWarps) {
    // ---- producer: one lane issues the TMA copies ----
    if (lane != 0 || p.debug) return;
    tile_produce<ND>(p, full_bar, empty_bar, coords, stages, ns);
    return;
  }

  // ---- consumers ----
  constexpr int RPT = tile_rows_per_thread(TIER);
  constexpr int V = 8 * RPT;
  const int cj = threadIdx.x & 7;         // columns 8 cj .. 8 cj + 7 of the tile
  const int rg = threadIdx.x >> 3;        // row group: rows RPT rg .. RPT rg + RPT - 1 of a pass
  const uint32_t* prog = c_prog[p.prog];
  if (p.debug) {
    // test hook: a wait that nothing satisfies must give up and report
    if (!mbar_wait(debug_bar, 0, p.timeout_ns) && lane == 0) atomicOr(p.err, kErrDebugWait);
    return;
  }
  StageRing ring;
  for (uint32_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ring.next(ns)) {
    const uint32_t s = ring.s, ph = ring.ph;
    if (!mbar_wait(full_bar + 8 * s, ph, p.timeout_ns)) {
      if (lane == 0) atomicOr(p.err, kErrConsumerWait);
      return;
    }
    const uint4 tcrd = lds128(coords + 16 * s);  // written by the producer with this stage
    const uint32_t tr = tcrd.x, tc = tcrd.y, b0 = tcrd.z, b1 = tcrd.w;
    const int64_t i0 = (int64_t)tr * kTileRows, j0 = (int64_t)tc * kTileCols;
    const uint32_t st = stages + s * p.stage_bytes;
#pragma unroll 1
    for (int pass = 0; pass < kTileRows / (32 * RPT); ++pass) {
      const int li = pass * 32 * RPT + RPT * rg;
      const int64_t i = i0 + li;
      const int64_t jc = j0 + cj * 8;
      if (i < p.rows && jc < p.cols) {
        const int64_t left = p.cols - jc;
        const bool fullc = left >= 8;
        const int nleft = fullc ? 8 : (int)left;
        uint32_t r[S][V];
#pragma unroll
        for (int j = 0; j < NL; ++j) {
          if (j < (int)p.n_loads) {
            const uint32_t at = st + p.load_off[j];
            if (p.in_trans[j]) {
              if (ND && p.in_bcast[j]) {
#pragma unroll
                for (int q = 0; q < RPT; ++q) {
                  const uint32_t v = read_bcast_col(at, p.in_dt[j], li + q);
#pragma unroll
                  for (int m = 0; m < 8; ++m) r[j][8 * q + m] = v;
                }
              } else if constexpr (TIER == kTier2 && ND) {
                // (the host splits only here: in the plain 2-D kernel and the
                // wider tiers a second read path cost more than it saved)
                if (p.in_split[j]) read_trans2_split(r[j], at, p.in_dt[j], li, cj);
                else read_trans2(r[j], at, p.in_dt[j], li, cj);
              } else if constexpr (RPT == 2) {
                read_trans2(r[j], at, p.in_dt[j], li, cj);
              } else {
                read_trans(r[j], at, p.in_dt[j], li, cj);
              }
            } else {
              const bool bc0 = ND && p.in_bcast[j];
              const int la = bc0 ? 0 : li;
              if constexpr (RPT == 2) {
                read_row2(r[j], at, p.in_dt[j], la, bc0 ? 0 : li + 1, cj);
              } else {
                read_row(r[j], at, p.in_dt[j], la, cj);
              }
            }
          }
        }
        if constexpr (RPT == 2) {
          TileStore2<ND> sto{{p, i, jc, fullc, nleft, b0, b1}, i + 1 < p.rows};
          run_program<TIER, V, EXT>(r, prog, p.scal, sto);
        } else {
          TileStore<ND> sto{p, i, jc, fullc, nleft, b0, b1};
          run_program<TIER, V, EXT>(r, prog, p.scal, sto);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar + 8 * s);
  }
}

cudaError_t CMDX_TILE_NAME(tile2d_upload_t)(int slot, const uint32_t* words, int n) {
  return cudaMemcpyToSymbol(c_prog, words, sizeof(uint32_t) * n, sizeof(uint32_t) * kMaxWords * slot);
}

// ---- host side ----------------------------------------------------------------

template <int TIER, bool ND, bool EXT>
static cudaError_t launch_tier(const Tile2dParams& p, cudaStream_t stream) {
  const size_t smem = (size_t)kBarrierBytes + (size_t)p.n_stages * p.stage_bytes;
  static DeviceCache grid_cache[kMaxStages + 1];  // (static storage: zero before first use)
  static DeviceCache attr_set;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set.get(dev)) {
    cudaError_t e = cudaFuncSetAttribute(tile2d_kernel<TIER, ND, EXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kBarrierBytes + 2 * kTileStageLimit + 4096);
    if (e != cudaSuccess) return e;
    attr_set.put(dev, 1);
  }
  // occupancy depends on the stage size; cached for the common size only
  const bool cache_ok = p.stage_bytes == 16384 && p.n_stages <= (uint32_t)kMaxStages;
  int full_grid = cache_ok ? grid_cache[p.n_stages].get(dev) : 0;
  if (full_grid == 0) {
    full_grid = persistent_grid(tile2d_kernel<TIER, ND, EXT>, kThreads, smem, INT64_MAX);
    if (cache_ok) grid_cache[p.n_stages].put(dev, full_grid);
  }
  const int grid = (int)(p.n_tiles < full_grid ? p.n_tiles : full_grid);
  return launch_pdl(tile2d_kernel<TIER, ND, EXT>, grid, kThreads, smem, stream, p);
}

cudaError_t CMDX_TILE_NAME(tile2d_launch_t)(const Tile2dParams& p, cudaStream_t stream) {
  return launch_tier<CMDX_TIER, CMDX_ND != 0, CMDX_EXT != 0>(p, stream);
}

}  // namespace cmdx
