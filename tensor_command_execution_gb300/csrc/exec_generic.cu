// exec_generic.cu - executor for any sizes/strides (rank <= 4 after merging,
// strides >= 0, including stride-0 broadcasts and permuted views).
//
// Each element's offset in every view is computed from its logical index as
// sum_k i_k * stride_k, with the multi-index taken from the row-major linear
// index (rocRoller, "Design Overview", section "Kernel Graph": Dimension nodes
// with size and stride, and the Flatten transform's row-major order). Lane l
// of a warp handles elements base + 32 v + l, so views that are contiguous in
// the innermost dim are still read with consecutive addresses across a warp.
//
// Compiled once per tier and op-set variant: CMDX_TIER and CMDX_EXT select
// the kernel this object holds.
#include "exec_common.cuh"

#if !defined(CMDX_TIER) || !defined(CMDX_EXT)
#error "exec_generic.cu is compiled per tier and variant, with -DCMDX_TIER=<0..4> -DCMDX_EXT=<0|1>"
#endif

namespace cmdx {

static __constant__ uint32_t c_prog[kMaxPrograms][kMaxWords];

// q = e / d with the divisor's precomputed multiply-high form.
__device__ __forceinline__ uint64_t fast_div(const FastDiv& f, uint64_t e) {
  const uint64_t t = __umul64hi(f.m, e);
  return (t + ((e - t) >> 1)) >> (f.l - 1);
}

// Offset of linear element e in a view with right-aligned strides st: the
// row-major multi-index of e dotted with the strides. The outermost dim of
// size > 1 takes what remains without a division (e < n bounds it), so a
// rank-1 view costs one multiply.
__device__ __forceinline__ int64_t gen_offset(const GenericParams& p, const int64_t* st, int64_t e) {
  int64_t off = 0;
  uint64_t rem = (uint64_t)e;
#pragma unroll
  for (int k = kMaxRank - 1; k > 0; --k) {
    if (k == (int)p.top) return off + (int64_t)rem * st[k];
    if (p.div[k].l == 0) continue;  // size-1 dim
    const uint64_t q = fast_div(p.div[k], rem);
    off += (int64_t)(rem - q * (uint64_t)p.div[k].d) * st[k];
    rem = q;
  }
  return off + (int64_t)rem * st[0];
}

// The row-major multi-index of linear element e, dims top .. kMaxRank - 1
// (c[k] for k < top stays 0): computed once per element and dotted with each
// view's strides by view_offset, so a launch with several loads divides once
// per element, not once per view.
__device__ __forceinline__ void gen_index(const GenericParams& p, int64_t e, int64_t (&c)[kMaxRank]) {
  uint64_t rem = (uint64_t)e;
#pragma unroll
  for (int k = kMaxRank - 1; k >= 0; --k) {
    c[k] = 0;
    if (k < (int)p.top) continue;
    if (k == (int)p.top || p.div[k].l == 0) {
      c[k] = k == (int)p.top ? (int64_t)rem : 0;
      if (k == (int)p.top) rem = 0;
      continue;
    }
    const uint64_t q = fast_div(p.div[k], rem);
    c[k] = (int64_t)(rem - q * (uint64_t)p.div[k].d);
    rem = q;
  }
}

__device__ __forceinline__ int64_t view_offset(const GenericParams& p, const int64_t (&c)[kMaxRank], const int64_t* st) {
  int64_t off = c[kMaxRank - 1] * st[kMaxRank - 1];
#pragma unroll
  for (int k = 0; k < kMaxRank - 1; ++k)
    if (k >= (int)p.top) off += c[k] * st[k];
  return off;
}

template <int V>
struct GenericStore {
  const GenericParams& p;
  int64_t base;
  int lane;

  template <int T>
  __device__ __forceinline__ void store(const uint32_t (&x)[V], uint32_t o) const {
    void* ptr = p.out[o];
    if constexpr (T == kStB1) {
      // one bit per element, at its row-major index (the view is dense):
      // the warp's 32 consecutive elements base + 32 v + lane make one word
      // (launches with packed bits have no gap)
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t e = base + 32 * v + lane;
        const uint32_t bits = __ballot_sync(0xffffffffu, e < p.n && x[v] != 0u);
        if (lane == 0 && base + 32 * v < p.n) __stcs(static_cast<unsigned int*>(ptr) + (base + 32 * v) / 32, bits);
      }
      return;
    }
    const int64_t* st = p.out_st[o];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int64_t e = base + 32 * v + lane;
      if (e < p.n) st_elem<T>(ptr, gen_offset(p, st, e < p.gap_at ? e : e + p.gap), x[v]);
    }
  }
};

template <int TIER, bool EXT>
__global__ void __launch_bounds__(256, tier_min_blocks(TIER)) generic_kernel(const __grid_constant__ GenericParams p) {
  constexpr int S = tier_slots(TIER);
  constexpr int V = tier_vec_strided(TIER);
  constexpr int NL = S < kMaxLoads ? S : kMaxLoads;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t* prog = c_prog[p.prog];
  pdl_wait();
  pdl_trigger();
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w * 32 * V < p.n; w += nwarps) {
    const int64_t base = w * 32 * V;
    uint32_t r[S][V];
    // every load of every view is issued before any is widened, so they are
    // all in flight at once (a widening right after each load would wait for
    // it before the next load issues)
    if (p.top == kMaxRank - 1) {
      // one dim: an element's offset in a view is one multiply
#pragma unroll
      for (int j = 0; j < NL; ++j) {
        if (j < (int)p.n_loads) {
#pragma unroll
          for (int v = 0; v < V; ++v) {
            const int64_t e = base + 32 * v + lane;
            r[j][v] = 0u;
            if (e < p.n)
              r[j][v] = ld_elem(p.in[j], p.in_dt[j], (e < p.gap_at ? e : e + p.gap) * p.in_st[j][kMaxRank - 1]);
          }
        }
      }
    } else {
      // several dims: the multi-index once per element, for every load
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t e = base + 32 * v + lane;
        int64_t c[kMaxRank];
        gen_index(p, e < p.gap_at ? e : e + p.gap, c);
#pragma unroll
        for (int j = 0; j < NL; ++j) {
          if (j < (int)p.n_loads) {
            r[j][v] = 0u;
            if (e < p.n) r[j][v] = ld_elem(p.in[j], p.in_dt[j], view_offset(p, c, p.in_st[j]));
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      if (j < (int)p.n_loads && (p.in_dt[j] == 1 || p.in_dt[j] == 2)) {
#pragma unroll
        for (int v = 0; v < V; ++v) r[j][v] = widen_any(p.in_dt[j], r[j][v]);
      }
    }
    GenericStore<V> st{p, base, lane};
    run_program<TIER, V, EXT>(r, prog, p.scal, st);
  }
}

cudaError_t CMDX_TIER_NAME(generic_upload_t)(int slot, const uint32_t* words, int n) {
  return cudaMemcpyToSymbol(c_prog, words, sizeof(uint32_t) * n, sizeof(uint32_t) * kMaxWords * slot);
}

template <int TIER, bool EXT>
static cudaError_t launch_tier(const GenericParams& p, cudaStream_t stream) {
  constexpr int V = tier_vec_strided(TIER);
  constexpr int kBlock = 256;
  static DeviceCache grid_cache;  // (static storage: zero before first use)
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t work_blocks = (p.n + (int64_t)kBlock * V - 1) / ((int64_t)kBlock * V);
  int full_grid = grid_cache.get(dev);
  if (full_grid == 0) {
    full_grid = persistent_grid(generic_kernel<TIER, EXT>, kBlock, 0, INT64_MAX);
    grid_cache.put(dev, full_grid);
  }
  const int grid = (int)(work_blocks < full_grid ? work_blocks : full_grid);
  return launch_pdl(generic_kernel<TIER, EXT>, grid, kBlock, 0, stream, p);
}

cudaError_t CMDX_TIER_NAME(generic_launch_t)(const GenericParams& p, cudaStream_t stream) {
  return launch_tier<CMDX_TIER, CMDX_EXT != 0>(p, stream);
}

}  // namespace cmdx
