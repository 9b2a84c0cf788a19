// exec_common.cuh - the register-slot interpreter shared by the executors.
//
// Every thread keeps V elements of each live value in registers ("slots").
// A program word selects one case of a jump table whose slot numbers are
// fixed in the code, so slots never need run-time register indexing (which
// would spill them to local memory). All threads of a launch run the same
// program, so the dispatch branch is warp-uniform. The loop is inline PTX
// (interp_asm.cuh, generated): in the 2-, 4- and 8-slot tiers one jump per
// word on (op, destination, source), each case updating its destination's
// registers in place, so the dispatch moves no data; in the 16- and 32-slot
// tiers two jumps per word, the first copying the source slot into staging
// registers, the second applying the op to the destination.
//
// rocRoller, "Design Overview": the program plays the part of the scheduled
// instructions generated from the KernelGraph (sections "Generating
// Instructions from a KernelGraph" and "Registers"); here it is interpreted by
// a hand-written kernel instead of being assembled per Command.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cmd_internal.h"
#include "interp_asm.cuh"

// The name of this object's entry point: CMDX_TIER_NAME(f_t) is f_t<T>e<E>
// for CMDX_TIER = T (0..3) and CMDX_EXT = E (0: the base op set, 1: extended,
// with division, comparisons, select and packed-bit stores).
#define CMDX_TIER_CAT2(a, b) a##b
#define CMDX_TIER_CAT(a, b) CMDX_TIER_CAT2(a, b)
// An object built with CMDX_OCC4=1 (a contiguous kernel sized for four
// resident CTAs per SM) appends o4; one built with CMDX_HALF16=1 (the
// contiguous 4-slot kernel at 16 elements per slot, for programs whose loads
// are all 2-byte) appends h16.
#ifndef CMDX_OCC4
#define CMDX_OCC4 0
#endif
#ifndef CMDX_HALF16
#define CMDX_HALF16 0
#endif
#if CMDX_OCC4
#define CMDX_TIER_NAME(f) CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(f, CMDX_TIER), e), CMDX_EXT), o4)
#elif CMDX_HALF16
#define CMDX_TIER_NAME(f) CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(f, CMDX_TIER), e), CMDX_EXT), h16)
#else
#define CMDX_TIER_NAME(f) CMDX_TIER_CAT(CMDX_TIER_CAT(CMDX_TIER_CAT(f, CMDX_TIER), e), CMDX_EXT)
#endif

namespace cmdx {

// ---- element operations on 32-bit slot words ------------------------------
// Float ops use the round-to-nearest-even intrinsics, which are never fused
// into a multiply-add; int ops are unsigned, i.e. modulo 2^32.
// minimumNumber / maximumNumber: min.f32 / max.f32 without .ftz return the
// number when one operand is NaN, order -0 below +0 and keep denormals.
__device__ __forceinline__ uint32_t fmin_num(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.f32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t fmax_num(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.f32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// int32 division truncating toward zero; x / 0 = -1, INT_MIN / -1 = INT_MIN.
__device__ __forceinline__ uint32_t idiv(uint32_t a, uint32_t b) {
  if (b == 0u) return 0xffffffffu;
  if (b == 0xffffffffu) return 0u - a;
  return (uint32_t)((int32_t)a / (int32_t)b);
}

template <int OP>
__device__ __forceinline__ uint32_t bin(uint32_t d, uint32_t x) {
  if constexpr (OP == kFAdd) return __float_as_uint(__fadd_rn(__uint_as_float(d), __uint_as_float(x)));
  if constexpr (OP == kFSub) return __float_as_uint(__fsub_rn(__uint_as_float(d), __uint_as_float(x)));
  if constexpr (OP == kFRsub) return __float_as_uint(__fsub_rn(__uint_as_float(x), __uint_as_float(d)));
  if constexpr (OP == kFMul) return __float_as_uint(__fmul_rn(__uint_as_float(d), __uint_as_float(x)));
  if constexpr (OP == kIAdd) return d + x;
  if constexpr (OP == kISub) return d - x;
  if constexpr (OP == kIRsub) return x - d;
  if constexpr (OP == kIMul) return d * x;
  if constexpr (OP == kFDiv) return __float_as_uint(__fdiv_rn(__uint_as_float(d), __uint_as_float(x)));
  if constexpr (OP == kFRdiv) return __float_as_uint(__fdiv_rn(__uint_as_float(x), __uint_as_float(d)));
  if constexpr (OP == kIDiv) return idiv(d, x);
  if constexpr (OP == kIRdiv) return idiv(x, d);
  if constexpr (OP == kFMin) return fmin_num(d, x);
  if constexpr (OP == kFMax) return fmax_num(d, x);
  if constexpr (OP == kIMin) return (int32_t)d < (int32_t)x ? d : x;
  if constexpr (OP == kIMax) return (int32_t)d > (int32_t)x ? d : x;
  return 0;
}

// Comparison c (CmpOp) of d with x: 1 or 0. Float relations are the IEEE
// ones (a NaN makes all but != false; -0 == +0).
__device__ __forceinline__ uint32_t cmp_rel(int c, uint32_t d, uint32_t x) {
  const float fd = __uint_as_float(d), fx = __uint_as_float(x);
  const int32_t id = (int32_t)d, ix = (int32_t)x;
  bool r;
  switch (c) {
    case kCFLt: r = fd < fx; break;
    case kCFLe: r = fd <= fx; break;
    case kCFGt: r = fd > fx; break;
    case kCFGe: r = fd >= fx; break;
    case kCFEq: r = fd == fx; break;
    case kCFNe: r = fd != fx; break;
    case kCILt: r = id < ix; break;
    case kCILe: r = id <= ix; break;
    case kCIGt: r = id > ix; break;
    case kCIGe: r = id >= ix; break;
    case kCIEq: r = d == x; break;
    case kCINe: r = d != x; break;
    case kCULt: r = d < x; break;
    case kCULe: r = d <= x; break;
    case kCUGt: r = d > x; break;
    default: r = d >= x; break;
  }
  return r ? 1u : 0u;
}

template <int OP>
__device__ __forceinline__ uint32_t un(uint32_t x) {
  if constexpr (OP == kFNeg) return x ^ 0x80000000u;  // IEEE negate: sign flip
  if constexpr (OP == kINeg) return 0u - x;
  if constexpr (OP == kFAbs) return x & 0x7fffffffu;
  if constexpr (OP == kIAbs) return (int32_t)x < 0 ? 0u - x : x;
  if constexpr (OP == kI2F) return __float_as_uint(__int2float_rn((int32_t)x));
  if constexpr (OP == kF2I) return (uint32_t)__float2int_rz(__uint_as_float(x));  // saturates, NaN -> 0
  return x;  // kMov
}

// ---- widening and narrowing ------------------------------------------------
__device__ __forceinline__ void widen_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  float2 f = __half22float2(h);
  lo = __float_as_uint(f.x);
  hi = __float_as_uint(f.y);
}
// bfloat16 is the upper half of a binary32 encoding: widening is a shift.
__device__ __forceinline__ void widen_bf16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = w << 16;
  hi = w & 0xffff0000u;
}
__device__ __forceinline__ uint32_t widen_f16(uint16_t h) {
  return __float_as_uint(__half2float(__ushort_as_half(h)));
}
__device__ __forceinline__ uint32_t widen_bf16(uint16_t h) { return uint32_t(h) << 16; }

__device__ __forceinline__ uint32_t narrow_f16x2(uint32_t lo, uint32_t hi) {
  __half2 h = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t narrow_bf16x2(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint16_t narrow_f16(uint32_t x) {
  return __half_as_ushort(__float2half_rn(__uint_as_float(x)));
}
__device__ __forceinline__ uint16_t narrow_bf16(uint32_t x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(x)));
}

// Widen one loaded element of type dt (raw bits) to a slot word.
__device__ __forceinline__ uint32_t widen_any(int dt, uint32_t raw) {
  if (dt == 1) return widen_f16((uint16_t)raw);
  if (dt == 2) return widen_bf16((uint16_t)raw);
  return raw;
}

// Streaming global accesses: every element is read or written once.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ uint2 ld_stream(const uint2* p) { return __ldcs(p); }
__device__ __forceinline__ uint32_t ld_stream(const uint32_t* p) { return __ldcs(reinterpret_cast<const unsigned int*>(p)); }
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint2* p, uint2 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint32_t* p, uint32_t v) { __stcs(reinterpret_cast<unsigned int*>(p), v); }
__device__ __forceinline__ void st_stream(uint16_t* p, uint16_t v) { __stcs(reinterpret_cast<unsigned short*>(p), v); }

// Load/store one raw element of type dt at element offset off.
__device__ __forceinline__ uint32_t ld_elem(const void* base, int dt, int64_t off) {
  if (dt == 1 || dt == 2) return __ldcs(reinterpret_cast<const unsigned short*>(base) + off);
  return __ldcs(reinterpret_cast<const unsigned int*>(base) + off);
}
template <int T>
__device__ __forceinline__ void st_elem(void* base, int64_t off, uint32_t x) {
  if constexpr (T == kStF16) __stcs(reinterpret_cast<unsigned short*>(base) + off, narrow_f16(x));
  else if constexpr (T == kStBF16) __stcs(reinterpret_cast<unsigned short*>(base) + off, narrow_bf16(x));
  else __stcs(reinterpret_cast<unsigned int*>(base) + off, x);
}

// ---- slot lists for the fused dispatch ----------------------------------------
#define CMDX_SA2(M, ...) M(0, __VA_ARGS__) M(1, __VA_ARGS__)
#define CMDX_SA4(M, ...) M(0, __VA_ARGS__) M(1, __VA_ARGS__) M(2, __VA_ARGS__) M(3, __VA_ARGS__)
#define CMDX_SA8(M, ...) CMDX_SA4(M, __VA_ARGS__) M(4, __VA_ARGS__) M(5, __VA_ARGS__) M(6, __VA_ARGS__) M(7, __VA_ARGS__)

#define CMDX_UNROLL _Pragma("unroll")

// store slot s as type t (case number relative to the first store case)
#define CMDX_ST_CASE(s_, t_)         \
  case (t_) * S + (s_):              \
    pol.template store<t_>(r[s_], aux); \
    break;

// packed-bit stores exist in the extended variant only (the base variant
// ends the program there; the host never launches that pairing)
#define CMDX_ST_CASE_B1(s_, t_)                                 \
  case kStB1 * S + (s_):                                        \
    if constexpr (EXT) pol.template store<kStB1>(r[s_], aux);   \
    else return;                                                \
    break;

#define CMDX_ST_CASES(SA)                                                                       \
  SA(CMDX_ST_CASE, kStF32) SA(CMDX_ST_CASE, kStF16) SA(CMDX_ST_CASE, kStBF16) SA(CMDX_ST_CASE, kStI32) \
  SA(CMDX_ST_CASE_B1, 0)

// Run the program in `prog` (constant memory) over the thread's slots. The
// compute words run inside the inline-PTX loop of interp_asm.cuh; each store
// word comes back here and is performed by Pol::store<T>(slot, out_index).
template <int S, int V, bool EXT, class Pol>
__device__ __forceinline__ void run_fused(uint32_t (&r)[S][V], const uint32_t* __restrict__ prog,
                                          const uint32_t* __restrict__ scal, Pol& pol) {
  // (in the base variant an extended word leaves the loop and ends the
  // program here, like the end word; the host never launches that pairing)
  static_assert(S == 2 || S == 4 || S == 8, "fused dispatch is generated for 2, 4 and 8 slots");
  uint32_t idx = 0;
#pragma unroll 1
  for (;;) {
    const uint32_t w = AsmInterp<S, V, EXT>::run(r, idx, prog, scal);
    const uint32_t c = (w & 0xffffu) - fz_store(S, 0, 0);
    if (c >= uint32_t(kNumSt) * S) return;  // the end word
    const uint32_t aux = w >> 16;
    if constexpr (S == 2) {
      switch (c) {
        CMDX_ST_CASES(CMDX_SA2)
        default: return;
      }
    } else if constexpr (S == 4) {
      switch (c) {
        CMDX_ST_CASES(CMDX_SA4)
        default: return;
      }
    } else {
      switch (c) {
        CMDX_ST_CASES(CMDX_SA8)
        default: return;
      }
    }
  }
}

// ---- wide dispatch (16 and 32 slots): fetch the source, then (op, dst) ------
#define CMDX_SA16(M, ...)                                                                 \
  CMDX_SA8(M, __VA_ARGS__) M(8, __VA_ARGS__) M(9, __VA_ARGS__) M(10, __VA_ARGS__)         \
  M(11, __VA_ARGS__) M(12, __VA_ARGS__) M(13, __VA_ARGS__) M(14, __VA_ARGS__) M(15, __VA_ARGS__)
#define CMDX_SA32(M, ...)                                                                 \
  CMDX_SA16(M, __VA_ARGS__) M(16, __VA_ARGS__) M(17, __VA_ARGS__) M(18, __VA_ARGS__)      \
  M(19, __VA_ARGS__) M(20, __VA_ARGS__) M(21, __VA_ARGS__) M(22, __VA_ARGS__)             \
  M(23, __VA_ARGS__) M(24, __VA_ARGS__) M(25, __VA_ARGS__) M(26, __VA_ARGS__)             \
  M(27, __VA_ARGS__) M(28, __VA_ARGS__) M(29, __VA_ARGS__) M(30, __VA_ARGS__) M(31, __VA_ARGS__)

#define CMDX_W_GET(s_, x_) \
  case s_: {               \
    CMDX_UNROLL for (int v = 0; v < V; ++v) y[v] = r[s_][v]; \
  } break;
#define CMDX_W_PUT(s_, x_) \
  case s_: {               \
    CMDX_UNROLL for (int v = 0; v < V; ++v) r[s_][v] = y[v]; \
  } break;

// y = slot s, and slot s = y, for a slot number known only at run time (a
// switch over the tier's slots, so the slots stay in registers).
template <int S, int V>
__device__ __forceinline__ void slot_get(const uint32_t (&r)[S][V], uint32_t s, uint32_t (&y)[V]) {
  if constexpr (S == 32) {
    switch (s) {
      CMDX_SA32(CMDX_W_GET, 0)
      default: break;
    }
  } else {
    switch (s) {
      CMDX_SA16(CMDX_W_GET, 0)
      default: break;
    }
  }
}
template <int S, int V>
__device__ __forceinline__ void slot_put(uint32_t (&r)[S][V], uint32_t s, const uint32_t (&y)[V]) {
  if constexpr (S == 32) {
    switch (s) {
      CMDX_SA32(CMDX_W_PUT, 0)
      default: break;
    }
  } else {
    switch (s) {
      CMDX_SA16(CMDX_W_PUT, 0)
      default: break;
    }
  }
}

// A wide tier (S = 16 or 32 slots): the arithmetic, min/max and unary words
// run in the inline-PTX loop of AsmWide (a jump on the source slot, then one
// on the op and destination); each word it returns (a store, the end, a
// division, comparison or select) is performed here and the loop re-entered.
template <int S, int V, bool EXT, class Pol>
__device__ __forceinline__ void run_wide(uint32_t (&r)[S][V], const uint32_t* __restrict__ prog,
                                         const uint32_t* __restrict__ scal, Pol& pol) {
  static_assert(S == 16 || S == 32, "the wide dispatch is generated for 16 and 32 slots");
  uint32_t pc = 0;
#pragma unroll 1
  for (;;) {
    const uint32_t w = AsmWide<S, V>::run(r, pc, prog, scal);
    const uint32_t kind = w >> 24;
    const uint32_t aux = w & 0xffu;
    const uint32_t base = kind & 0x3fu;
    if (base == kWEnd) return;
    uint32_t x[V];
    if (kind & kWScalar) {
      const uint32_t k = scal[aux];
      CMDX_UNROLL for (int v = 0; v < V; ++v) x[v] = k;
    } else {
      slot_get<S, V>(r, (w >> 8) & 0xffu, x);
    }
    const uint32_t d = (w >> 16) & 0xffu;
    if (base >= kWBin0 + kFDiv && base <= kWBin0 + kIRdiv) {
      // the division ops (kFDiv, kFRdiv, kIDiv, kIRdiv are consecutive): one
      // body for every destination, fetch, divide, write back; the base
      // variant ends the program (the host never launches that pairing)
      if constexpr (!EXT) return;
      uint32_t y[V];
      slot_get<S, V>(r, d, y);
      const uint32_t op = base - kWBin0;
      CMDX_UNROLL for (int v = 0; v < V; ++v) {
        const bool rev = op == kFRdiv || op == kIRdiv;
        const uint32_t a = rev ? x[v] : y[v], b = rev ? y[v] : x[v];
        y[v] = op >= kIDiv ? idiv(a, b) : bin<kFDiv>(a, b);
      }
      slot_put<S, V>(r, d, y);
      continue;
    }
    if (base >= kWCmp0 && base < kWCmp0 + kNumCmp) {
      // comparisons: one body for every destination, like the divisions
      if constexpr (!EXT) return;
      uint32_t y[V];
      slot_get<S, V>(r, d, y);
      CMDX_UNROLL for (int v = 0; v < V; ++v) y[v] = cmp_rel((int)(base - kWCmp0), y[v], x[v]);
      slot_put<S, V>(r, d, y);
      continue;
    }
    if (base == kWSDiv0 || base == kWSDiv0 + 1) {
      // division by a scalar through the derived constants at aux..: the fast
      // sequence when every element of the warp is in range, else the
      // general division (the same arithmetic as the fused cases)
      if constexpr (!EXT) return;
      uint32_t y[V];
      slot_get<S, V>(r, d, y);
      if (base == kWSDiv0) {
        const float sv = __uint_as_float(scal[aux]), rv = __uint_as_float(scal[aux + 1]);
        bool ok = rv != 0.0f;
        CMDX_UNROLL for (int v = 0; v < V; ++v) {
          const float a = fabsf(__uint_as_float(y[v]));
          ok = ok && a >= 0x1p-60f && a <= 0x1p60f;
        }
        if (__all_sync(__activemask(), ok)) {
          CMDX_UNROLL for (int v = 0; v < V; ++v) {
            const float xv = __uint_as_float(y[v]);
            float q = __fmul_rn(xv, rv);
            q = __fmaf_rn(__fmaf_rn(-q, sv, xv), rv, q);
            q = __fmaf_rn(__fmaf_rn(-q, sv, xv), rv, q);
            y[v] = __float_as_uint(q);
          }
        } else {
          CMDX_UNROLL for (int v = 0; v < V; ++v) y[v] = bin<kFDiv>(y[v], scal[aux]);
        }
      } else {
        const uint32_t sh = scal[aux + 2];
        if (sh & kSDivSlow) {
          CMDX_UNROLL for (int v = 0; v < V; ++v) y[v] = idiv(y[v], scal[aux]);
        } else {
          const int32_t m = (int32_t)scal[aux + 1], ds = (int32_t)scal[aux] >> 31;
          CMDX_UNROLL for (int v = 0; v < V; ++v) {
            const int32_t n = (int32_t)y[v];
            int32_t q = n + __mulhi(m, n);
            q = (q >> sh) - (n >> 31);
            y[v] = (uint32_t)((q ^ ds) - ds);
          }
        }
      }
      slot_put<S, V>(r, d, y);
      continue;
    }
    if (base == kWSel) {
      // d = X != 0 ? d : x, X the staging slot S - 1
      if constexpr (!EXT) return;
      uint32_t y[V];
      slot_get<S, V>(r, d, y);
      CMDX_UNROLL for (int v = 0; v < V; ++v) y[v] = r[S - 1][v] != 0u ? y[v] : x[v];
      slot_put<S, V>(r, d, y);
      continue;
    }
    if (base >= kWStore0 && base < kWStore0 + kNumSt) {
      switch (base - kWStore0) {
        case kStF32: pol.template store<kStF32>(x, aux); break;
        case kStB1:
          if constexpr (EXT) pol.template store<kStB1>(x, aux);
          else return;
          break;
        case kStF16: pol.template store<kStF16>(x, aux); break;
        case kStBF16: pol.template store<kStBF16>(x, aux); break;
        default: pol.template store<kStI32>(x, aux); break;
      }
      continue;
    }
    return;  // (not reached: AsmWide runs every other kind)
  }
}

template <int TIER, int V, bool EXT, class Pol>
__device__ __forceinline__ void run_program(uint32_t (&r)[tier_slots(TIER)][V], const uint32_t* prog,
                                            const uint32_t* scal, Pol& pol) {
  if constexpr (tier_wide(TIER)) run_wide<tier_slots(TIER), V, EXT>(r, prog, scal, pol);
  else run_fused<tier_slots(TIER), V, EXT>(r, prog, scal, pol);
}

// ---- element-to-lane map of the contiguous and generic executors --------------
// A warp covers 32*V consecutive logical elements. Lane l holds NG groups of G
// consecutive elements; group h starts at h*32*G + l*G. With G = 4, each
// group of a 4-byte tensor is one 16-byte access and a warp's access to one
// group is 512 contiguous bytes.
template <int V>
struct LaneMap {
  static constexpr int G = V < 4 ? V : 4;
  static constexpr int NG = V / G;
  static constexpr int W = 32 * V;
};

// ---- programmatic dependent launch ------------------------------------------
// Every executor launch may begin while the previous kernel on its stream is
// still running: its CTAs are scheduled early, and each one first waits
// (griddepcontrol.wait) until that kernel has completed and its memory is
// visible, so no data access overlaps it and a Command that reads what the
// previous one wrote stays correct. Each CTA then lets the next launch start
// (griddepcontrol.launch_dependents). What overlaps is launch processing and
// CTA scheduling, which dominate small launches. Without the launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <class K, class P>
inline cudaError_t launch_pdl(K kernel, int grid, int block, size_t smem, cudaStream_t stream, const P& params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, params);
}

// A value computed once per device by host code (a grid size, a flag that a
// kernel attribute is set), read and written from any host thread: relaxed
// atomics suffice, since every thread that computes it computes the same
// value and a race only repeats the computation. Zero means "not yet"; a
// device index outside the table is never cached.
struct DeviceCache {
  static constexpr int kDevices = 64;
  std::atomic<int> v[kDevices];
  int get(int dev) const { return dev >= 0 && dev < kDevices ? v[dev].load(std::memory_order_relaxed) : 0; }
  void put(int dev, int x) {
    if (dev >= 0 && dev < kDevices) v[dev].store(x, std::memory_order_relaxed);
  }
};

// Grid size for a persistent grid-stride kernel: enough CTAs to fill the
// device at the kernel's occupancy, and no more than the work needs.
template <class K>
inline int persistent_grid(K kernel, int block, size_t smem, int64_t work_blocks) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, smem);
  if (per_sm < 1) per_sm = 1;
  if (sms < 1) sms = 1;
  int64_t g = (int64_t)sms * per_sm;
  if (work_blocks < g) g = work_blocks;
  return g < 1 ? 1 : (int)g;
}

}  // namespace cmdx
