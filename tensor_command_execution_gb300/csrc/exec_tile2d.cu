// exec_tile2d.cu - 2-D strided executor for views that are row-direct
// (element (i, j) at i*ld + j) or transposed (element (i, j) at i + j*ld).
//
// A CTA of 256 threads walks 64 x 64 tiles of the logical index space. Each
// thread owns V (8 or 4) consecutive columns of one row per pass, so
// row-direct loads and every store are vector accesses and a warp touches
// whole 128-byte (or larger) row segments. A transposed view is read along its physical
// rows (logical columns), which are contiguous in the logical row index: the
// tile's 64 physical row segments are copied into shared memory with 16-byte
// loads and then read transposed. The stage's 16-byte chunks are swizzled by
// XOR with (physical row / 8) mod 8, so the column groups a warp reads at
// once fall in distinct banks (at most two-way for V = 4) and the 16-byte
// stage writes stay aligned.
//
// rocRoller, "Design Overview", section "Kernel Graph": the coordinate
// transforms map each logical index to a tensor offset through sizes and
// strides; tiling and the shared-memory transpose are how this executor
// makes those transforms coalesce on the GPU (the pages' own generator stages
// tiles through LDS on AMD hardware).
#include "exec_common.cuh"

namespace cmdx {

static __constant__ uint32_t c_prog[kMaxPrograms][kMaxWords];

constexpr int kStageBytes = kTileRows * kTileCols * 4;  // one stage, sized for 4-byte elements
static_assert(kTileRows == 64 && kTileCols == 64, "the thread map below assumes 64 x 64 tiles");

// Copy the tile's physical rows of a transposed view into a stage.
__device__ __forceinline__ void stage_tile(unsigned char* stage, const void* base, int dt, int64_t ld,
                                           int64_t i0, int64_t j0, int64_t rows, int64_t cols, bool full, int tid) {
  const int es = (dt == 1 || dt == 2) ? 2 : 4;
  const int chunks_per_row = kTileRows * es / 16;  // 8 (2-byte) or 16 (4-byte)
  const int elems_per_chunk = 16 / es;
  const int n_chunks = kTileCols * chunks_per_row;
  for (int c = tid; c < n_chunks; c += 256) {
    const int q = c / chunks_per_row;     // physical row in the tile = logical column j0 + q
    const int ch = c - q * chunks_per_row;
    unsigned char* dst = stage + q * (kTileRows * es) + ((ch ^ ((q >> 3) & 7)) << 4);
    const int64_t i = i0 + (int64_t)ch * elems_per_chunk;
    const int64_t j = j0 + q;
    if (full) {
      const unsigned char* src = static_cast<const unsigned char*>(base) + (j * ld + i) * es;
      *reinterpret_cast<uint4*>(dst) = ld_stream(reinterpret_cast<const uint4*>(src));
    } else {
      if (es == 2) {
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          v[e] = (j < cols && i + e < rows) ? (uint16_t)ld_elem(base, dt, j * ld + i + e) : (uint16_t)0;
        uint4 w;
        w.x = v[0] | (uint32_t)v[1] << 16; w.y = v[2] | (uint32_t)v[3] << 16;
        w.z = v[4] | (uint32_t)v[5] << 16; w.w = v[6] | (uint32_t)v[7] << 16;
        *reinterpret_cast<uint4*>(dst) = w;
      } else {
        uint32_t v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = (j < cols && i + e < rows) ? ld_elem(base, dt, j * ld + i + e) : 0u;
        *reinterpret_cast<uint4*>(dst) = make_uint4(v[0], v[1], v[2], v[3]);
      }
    }
  }
}

// Thread map of a 64 x 64 tile for V columns per thread.
template <int V>
struct TileMap {
  static constexpr int TPR = kTileCols / V;        // threads per tile row
  static constexpr int RPP = 256 / TPR;            // rows per pass
  static constexpr int PASSES = kTileRows / RPP;
};

// Read logical (li, V*cj + k), k < V, from a stage and widen.
template <int V>
__device__ __forceinline__ void read_stage(uint32_t (&x)[V], const unsigned char* stage, int dt, int li, int cj) {
  const int es = (dt == 1 || dt == 2) ? 2 : 4;
  const int elems_per_chunk = 16 / es;
  const int ch = li / elems_per_chunk;
  const int within = (li - ch * elems_per_chunk) * es;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int q = V * cj + k;  // physical row of the stage
    const unsigned char* at = stage + q * (kTileRows * es) + ((ch ^ ((q >> 3) & 7)) << 4) + within;
    if (es == 2) {
      const uint16_t h = *reinterpret_cast<const uint16_t*>(at);
      x[k] = dt == 1 ? widen_f16(h) : widen_bf16(h);
    } else {
      x[k] = *reinterpret_cast<const uint32_t*>(at);
    }
  }
}

// Row-direct load of V consecutive columns.
template <int V>
__device__ __forceinline__ void row_load(uint32_t (&x)[V], const void* base, int dt, int64_t off, bool full,
                                         int ncols_left) {
  if (full) {
    if (dt == 0 || dt == 3) {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(base) + off);
#pragma unroll
      for (int h = 0; h < V / 4; ++h) {
        const uint4 a = ld_stream(p + h);
        x[4 * h] = a.x; x[4 * h + 1] = a.y; x[4 * h + 2] = a.z; x[4 * h + 3] = a.w;
      }
    } else {
      uint32_t w[V / 2];
      if constexpr (V == 8) {
        const uint4 a = ld_stream(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      } else {
        const uint2 a = ld_stream(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off));
        w[0] = a.x; w[1] = a.y;
      }
#pragma unroll
      for (int h = 0; h < V / 2; ++h) {
        if (dt == 1) widen_f16x2(w[h], x[2 * h], x[2 * h + 1]);
        else widen_bf16x2(w[h], x[2 * h], x[2 * h + 1]);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < V; ++k) x[k] = k < ncols_left ? widen_any(dt, ld_elem(base, dt, off + k)) : 0u;
  }
}

template <int V>
struct TileStore {
  const Tile2dParams& p;
  int64_t i, j;
  bool full;
  int ncols_left;

  template <int T>
  __device__ __forceinline__ void store(const uint32_t (&x)[V], uint32_t o) const {
    void* base = p.out[o];
    const int64_t off = i * p.out_ld[o] + j;
    if (full) {
      if constexpr (T == kStF32 || T == kStI32) {
        uint4* q = reinterpret_cast<uint4*>(static_cast<uint32_t*>(base) + off);
#pragma unroll
        for (int h = 0; h < V / 4; ++h) st_stream(q + h, make_uint4(x[4 * h], x[4 * h + 1], x[4 * h + 2], x[4 * h + 3]));
      } else {
        uint32_t w[V / 2];
#pragma unroll
        for (int h = 0; h < V / 2; ++h)
          w[h] = T == kStF16 ? narrow_f16x2(x[2 * h], x[2 * h + 1]) : narrow_bf16x2(x[2 * h], x[2 * h + 1]);
        if constexpr (V == 8)
          st_stream(reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + off), make_uint4(w[0], w[1], w[2], w[3]));
        else
          st_stream(reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + off), make_uint2(w[0], w[1]));
      }
    } else {
#pragma unroll
      for (int k = 0; k < V; ++k)
        if (k < ncols_left) st_elem<T>(base, off + k, x[k]);
    }
  }
};

template <int TIER>
__global__ void __launch_bounds__(256, tier_min_blocks(TIER)) tile2d_kernel(const __grid_constant__ Tile2dParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int S = tier_slots(TIER);
  constexpr int V = tier_vec_strided(TIER);
  static_assert(V == 4 || V == 8, "the tile executor keeps 4 or 8 columns per thread");
  using TM = TileMap<V>;
  constexpr int NL = S < kMaxLoads ? S : kMaxLoads;
  const int tid = threadIdx.x;
  const int cj = tid % TM::TPR;  // column group: columns V cj .. V cj + V - 1 of the tile
  const int ri = tid / TM::TPR;  // row within a pass
  const uint32_t* prog = c_prog[p.prog];
  for (int64_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
    const int64_t tr = t / p.tiles_c;
    const int64_t i0 = tr * kTileRows, j0 = (t - tr * p.tiles_c) * kTileCols;
    const bool full_tile = i0 + kTileRows <= p.rows && j0 + kTileCols <= p.cols;
    if (p.n_trans) {
      __syncthreads();  // the previous tile's stage readers are done
#pragma unroll
      for (int j = 0; j < NL; ++j)
        if (j < (int)p.n_loads && p.in_stage[j] >= 0)
          stage_tile(smem + p.in_stage[j] * kStageBytes, p.in[j], p.in_dt[j], p.in_ld[j], i0, j0, p.rows, p.cols,
                     full_tile, tid);
      __syncthreads();
    }
#pragma unroll 1
    for (int pass = 0; pass < TM::PASSES; ++pass) {
      const int li = pass * TM::RPP + ri;
      const int64_t i = i0 + li;
      const int64_t jc = j0 + cj * V;
      if (i >= p.rows || jc >= p.cols) continue;
      const int64_t left = p.cols - jc;
      const bool full = left >= V;
      const int ncols_left = full ? V : (int)left;
      uint32_t r[S][V];
#pragma unroll
      for (int j = 0; j < NL; ++j) {
        if (j < (int)p.n_loads) {
          if (p.in_stage[j] >= 0) read_stage<V>(r[j], smem + p.in_stage[j] * kStageBytes, p.in_dt[j], li, cj);
          else row_load<V>(r[j], p.in[j], p.in_dt[j], i * p.in_ld[j] + jc, full, ncols_left);
        }
      }
      TileStore<V> st{p, i, jc, full, ncols_left};
      run_program<TIER, V>(r, prog, p.scal, st);
    }
  }
}

cudaError_t tile2d_upload(int slot, const uint32_t* words, int n) {
  return cudaMemcpyToSymbol(c_prog, words, sizeof(uint32_t) * n, sizeof(uint32_t) * kMaxWords * slot);
}

template <int TIER>
static cudaError_t launch_tier(const Tile2dParams& p, cudaStream_t stream) {
  constexpr int kBlock = 256;
  const size_t smem = (size_t)p.n_trans * kStageBytes;
  static int grid_cache[64][5] = {};
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cacheable = dev >= 0 && dev < 64 && p.n_trans <= 4;
  if (cacheable && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tile2d_kernel<TIER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         4 * kStageBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int full_grid = cacheable ? grid_cache[dev][p.n_trans] : 0;
  if (full_grid == 0) {
    full_grid = persistent_grid(tile2d_kernel<TIER>, kBlock, smem, INT64_MAX);
    if (cacheable) grid_cache[dev][p.n_trans] = full_grid;
  }
  const int grid = (int)(p.n_tiles < full_grid ? p.n_tiles : full_grid);
  tile2d_kernel<TIER><<<grid, kBlock, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t tile2d_launch(int tier, const Tile2dParams& p, cudaStream_t stream) {
  switch (tier) {
    case kTier4: return launch_tier<kTier4>(p, stream);
    default: return launch_tier<kTier8>(p, stream);
  }
}

}  // namespace cmdx
