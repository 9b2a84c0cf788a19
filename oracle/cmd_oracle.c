/*
 * cmd_oracle.c - plain, slow CPU oracle for fused Command execution.
 *
 * TEST INFRASTRUCTURE: see cmd_oracle.h for who may use it and for the
 * readings of the pages it follows. Build with -ffp-contract=off and without
 * fast-math (a compiler that contracts a*b+c into one fused op, or flushes
 * denormals, would no longer compute the definition).
 */
#include "cmd_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- bits <-> values --------------------------------------------------- */

static float as_float(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint32_t as_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

/* ---- E operations (rocRoller Design Overview, "Operations": the T_Execute
 * block's E_ ops act elementwise on vectors or scalars) ------------------- */

/* Float E ops: exact result in binary64 (the product of two 24-bit
 * significands is exact; a sum is rounded to 53 bits), then one rounding to
 * binary32 by the C conversion, which rounds to nearest even. */
uint32_t orc_fadd(uint32_t x, uint32_t y) {
  double r = (double)as_float(x) + (double)as_float(y);
  return as_bits((float)r);
}

uint32_t orc_fsub(uint32_t x, uint32_t y) {
  double r = (double)as_float(x) - (double)as_float(y);
  return as_bits((float)r);
}

uint32_t orc_fmul(uint32_t x, uint32_t y) {
  double r = (double)as_float(x) * (double)as_float(y);
  return as_bits((float)r);
}

/* Negation is the IEEE 754 sign flip. */
uint32_t orc_fneg(uint32_t x) { return x ^ 0x80000000u; }

/* int32 E ops: two's complement, i.e. arithmetic modulo 2^32 on the bits. */
uint32_t orc_iadd(uint32_t x, uint32_t y) { return (uint32_t)(x + y); }
uint32_t orc_isub(uint32_t x, uint32_t y) { return (uint32_t)(x - y); }
uint32_t orc_imul(uint32_t x, uint32_t y) {
  return (uint32_t)((uint64_t)x * (uint64_t)y);
}
uint32_t orc_ineg(uint32_t x) { return (uint32_t)(0u - x); }

/* Division: the binary64 quotient rounded once more to binary32 (innocuous
 * for division as for + - x: Figueroa's condition 53 >= 2*24 + 2 holds). */
uint32_t orc_fdiv(uint32_t x, uint32_t y) {
  double r = (double)as_float(x) / (double)as_float(y);
  return as_bits((float)r);
}

uint32_t orc_idiv(uint32_t x, uint32_t y) {
  int32_t a = (int32_t)x, b = (int32_t)y;
  if (b == 0) return 0xffffffffu;                 /* x / 0 = -1 */
  if (a == INT32_MIN && b == -1) return x;        /* INT_MIN / -1 = INT_MIN */
  return (uint32_t)(a / b);                       /* C truncates toward zero */
}

/* minimumNumber / maximumNumber (IEEE 754-2019 section 9.6). */
uint32_t orc_fmin(uint32_t x, uint32_t y) {
  float a = as_float(x), b = as_float(y);
  if (isnan(a)) return y;
  if (isnan(b)) return x;
  if (a < b) return x;
  if (b < a) return y;
  return signbit(a) ? x : y; /* equal: for zeros the negative one is smaller */
}

uint32_t orc_fmax(uint32_t x, uint32_t y) {
  float a = as_float(x), b = as_float(y);
  if (isnan(a)) return y;
  if (isnan(b)) return x;
  if (a > b) return x;
  if (b > a) return y;
  return signbit(a) ? y : x;
}

uint32_t orc_imin(uint32_t x, uint32_t y) { return (int32_t)x < (int32_t)y ? x : y; }
uint32_t orc_imax(uint32_t x, uint32_t y) { return (int32_t)x > (int32_t)y ? x : y; }

uint32_t orc_fabs(uint32_t x) { return x & 0x7fffffffu; }
uint32_t orc_iabs(uint32_t x) { return ((int32_t)x < 0) ? (uint32_t)(0u - x) : x; }

/* int32 -> binary32: the exact value in binary64, rounded once. */
uint32_t orc_i2f(uint32_t x) { return as_bits((float)(double)(int32_t)x); }

/* binary32 -> int32: truncate toward zero, saturate, NaN -> 0. */
uint32_t orc_f2i(uint32_t x) {
  double v = (double)as_float(x);
  if (isnan(v)) return 0u;
  if (v >= 2147483648.0) return 0x7fffffffu;
  if (v <= -2147483649.0) return 0x80000000u;
  return (uint32_t)(int32_t)trunc(v);
}

/* Comparisons: 1 when the relation holds, else 0. Floats compare as IEEE
 * values (C's relational operators on float are the IEEE comparisons: a
 * NaN operand makes every one false but !=); ints as signed or unsigned
 * 32-bit numbers. */
uint32_t orc_compare(int32_t kind, int32_t is_int, uint32_t x, uint32_t y) {
  if (kind >= ORC_ULT) {
    switch (kind) {
      case ORC_ULT: return x < y;
      case ORC_ULE: return x <= y;
      case ORC_UGT: return x > y;
      default: return x >= y;
    }
  }
  if (is_int) {
    int32_t a = (int32_t)x, b = (int32_t)y;
    switch (kind) {
      case ORC_LT: return a < b;
      case ORC_LE: return a <= b;
      case ORC_GT: return a > b;
      case ORC_GE: return a >= b;
      case ORC_EQ: return a == b;
      default: return a != b;
    }
  }
  float a = as_float(x), b = as_float(y);
  switch (kind) {
    case ORC_LT: return a < b;
    case ORC_LE: return a <= b;
    case ORC_GT: return a > b;
    case ORC_GE: return a >= b;
    case ORC_EQ: return a == b;
    default: return a != b;
  }
}

/* ---- conversions ------------------------------------------------------- */

/* Round a non-negative finite value v (exactly representable in binary64)
 * to the nearest multiple of 2^q, ties to the even multiple. */
static double round_to_quantum(double v, int q) {
  double m = ldexp(v, -q);       /* exact: scaling by a power of two */
  double fl = floor(m);
  double fr = m - fl;            /* exact: m has at most 24 significant bits */
  if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  return ldexp(fl, q);
}

/* Round binary32 value bits to a binary format with p significand bits
 * (including the implicit one), minimum normal exponent emin and exponent
 * bias, and return the encoding of the rounded magnitude (sign excluded).
 * Overflow (rounded value >= 2^(emax+1)) gives the infinity encoding. */
static uint32_t round_magnitude(uint32_t xb, int p, int emin, int emax) {
  double v = fabs((double)as_float(xb));
  if (v == 0.0) return 0u;
  int e;
  frexp(v, &e);                  /* v = f * 2^e with f in [0.5, 1) */
  int E = e - 1;                 /* 2^E <= v < 2^(E+1) */
  int q = (E >= emin) ? (E - (p - 1)) : (emin - (p - 1));
  double r = round_to_quantum(v, q);
  int frac_bits = p - 1;
  uint32_t exp_all_ones = (uint32_t)(2 * emax + 1); /* biased exponent of inf */
  if (r >= ldexp(1.0, emax + 1)) return exp_all_ones << frac_bits;
  if (r < ldexp(1.0, emin)) {
    /* subnormal: significand = r / 2^(emin - (p-1)), biased exponent 0 */
    return (uint32_t)ldexp(r, -(emin - (p - 1)));
  }
  frexp(r, &e);
  E = e - 1;
  uint32_t sig = (uint32_t)ldexp(r, -(E - (p - 1))); /* in [2^(p-1), 2^p) */
  uint32_t frac = sig - (1u << frac_bits);
  uint32_t biased = (uint32_t)(E + emax);            /* bias = emax */
  return (biased << frac_bits) | frac;
}

/* binary32 -> binary16: p = 11, emin = -14, emax = 15. */
uint16_t orc_f32_to_f16(uint32_t x) {
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ax = x & 0x7fffffffu;
  if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7e00u); /* NaN -> quiet NaN */
  if (ax == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | round_magnitude(x, 11, -14, 15));
}

/* binary32 -> bfloat16: p = 8, emin = -126, emax = 127. */
uint16_t orc_f32_to_bf16(uint32_t x) {
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ax = x & 0x7fffffffu;
  if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7fc0u); /* NaN -> quiet NaN */
  if (ax == 0x7f800000u) return (uint16_t)(sign | 0x7f80u);
  return (uint16_t)(sign | round_magnitude(x, 8, -126, 127));
}

/* binary16 -> binary32, exact. */
uint32_t orc_f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  int E = (h >> 10) & 0x1f;
  int F = h & 0x3ff;
  if (E == 31) return sign | (F ? 0x7fc00000u : 0x7f800000u);
  double v = (E == 0) ? ldexp((double)F, -24) : ldexp((double)(1024 + F), E - 25);
  return sign | as_bits((float)v); /* exact: at most 11 significant bits */
}

/* bfloat16 is by definition the upper half of a binary32 encoding. */
uint32_t orc_bf16_to_f32(uint16_t h) { return ((uint32_t)h) << 16; }

void orc_f32_to_f16_n(const uint32_t* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

void orc_f32_to_bf16_n(const uint32_t* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

/* ---- the Command walk -------------------------------------------------- */

enum { CLS_FLOAT = 0, CLS_INT = 1 };

static size_t elem_size(int dtype) {
  return (dtype == ORC_F16 || dtype == ORC_BF16) ? 2u : 4u;
}

static int operand_ok(const orc_command* c, int32_t tag, int t) {
  return tag >= 0 && tag < t && c->ops[tag].kind != ORC_STORE;
}

/* Value class of every tag; checks operand classes and store types. */
static int classify(const orc_command* c, int* cls) {
  for (int t = 0; t < c->n_ops; ++t) {
    const orc_op* op = &c->ops[t];
    switch (op->kind) {
      case ORC_LOAD_TENSOR:
        if (op->dtype < ORC_F32 || op->dtype > ORC_I32) return ORC_ETYPE;
        cls[t] = (op->dtype == ORC_I32) ? CLS_INT : CLS_FLOAT;
        break;
      case ORC_LOAD_SCALAR:
        if (op->dtype != ORC_F32 && op->dtype != ORC_I32) return ORC_ETYPE;
        cls[t] = (op->dtype == ORC_I32) ? CLS_INT : CLS_FLOAT;
        break;
      case ORC_ADD:
      case ORC_SUB:
      case ORC_MUL:
        if (op->a < 0 || op->a >= t || op->b < 0 || op->b >= t) return ORC_EBAD;
        if (c->ops[op->a].kind == ORC_STORE || c->ops[op->b].kind == ORC_STORE) return ORC_EBAD;
        if (cls[op->a] != cls[op->b]) return ORC_ETYPE;
        cls[t] = cls[op->a];
        break;
      case ORC_DIV:
      case ORC_MIN:
      case ORC_MAX:
        if (op->a < 0 || op->a >= t || op->b < 0 || op->b >= t) return ORC_EBAD;
        if (c->ops[op->a].kind == ORC_STORE || c->ops[op->b].kind == ORC_STORE) return ORC_EBAD;
        if (cls[op->a] != cls[op->b]) return ORC_ETYPE;
        cls[t] = cls[op->a];
        break;
      case ORC_NEG:
      case ORC_ABS:
      case ORC_TO_F32:
      case ORC_TO_I32:
        if (op->a < 0 || op->a >= t) return ORC_EBAD;
        if (c->ops[op->a].kind == ORC_STORE) return ORC_EBAD;
        cls[t] = op->kind == ORC_TO_F32 ? CLS_FLOAT : op->kind == ORC_TO_I32 ? CLS_INT : cls[op->a];
        break;
      case ORC_LT:
      case ORC_LE:
      case ORC_GT:
      case ORC_GE:
      case ORC_EQ:
      case ORC_NE:
      case ORC_ULT:
      case ORC_ULE:
      case ORC_UGT:
      case ORC_UGE:
        if (!operand_ok(c, op->a, t) || !operand_ok(c, op->b, t)) return ORC_EBAD;
        if (cls[op->a] != cls[op->b]) return ORC_ETYPE;
        if (op->kind >= ORC_ULT && cls[op->a] != CLS_INT) return ORC_ETYPE;
        cls[t] = CLS_INT;
        break;
      case ORC_SELECT:
        if (!operand_ok(c, op->a, t) || !operand_ok(c, op->b, t) || !operand_ok(c, op->c, t))
          return ORC_EBAD;
        if (cls[op->a] != cls[op->b] || cls[op->c] != CLS_INT) return ORC_ETYPE;
        cls[t] = cls[op->a];
        break;
      case ORC_STORE:
        if (op->a < 0 || op->a >= t) return ORC_EBAD;
        if (c->ops[op->a].kind == ORC_STORE) return ORC_EBAD;
        if (op->dtype < ORC_F32 || op->dtype > ORC_B1) return ORC_ETYPE;
        if ((op->dtype == ORC_I32 || op->dtype == ORC_B1) != (cls[op->a] == CLS_INT)) return ORC_ETYPE;
        cls[t] = -1;
        break;
      default:
        return ORC_EBAD;
    }
  }
  return ORC_OK;
}

/* Element offset of a logical multi-index in a view: sum of index * stride. */
static int64_t view_offset(const orc_op* op, const int64_t* idx, int rank) {
  int64_t off = 0;
  for (int k = 0; k < rank; ++k) off += idx[k] * op->strides[k];
  return off;
}

static uint32_t load_elem(const orc_op* op, int64_t off) {
  const char* base = (const char*)op->ptr + off * (int64_t)elem_size(op->dtype);
  switch (op->dtype) {
    case ORC_F16: {
      uint16_t h;
      memcpy(&h, base, 2);
      return orc_f16_to_f32(h);
    }
    case ORC_BF16: {
      uint16_t h;
      memcpy(&h, base, 2);
      return orc_bf16_to_f32(h);
    }
    default: {
      uint32_t u;
      memcpy(&u, base, 4);
      return u;
    }
  }
}

/* Convert a value to a store's element type, writing elem_size bytes. */
static void convert_store(int dtype, uint32_t v, void* dst) {
  if (dtype == ORC_F16) {
    uint16_t h = orc_f32_to_f16(v);
    memcpy(dst, &h, 2);
  } else if (dtype == ORC_BF16) {
    uint16_t h = orc_f32_to_bf16(v);
    memcpy(dst, &h, 2);
  } else {
    memcpy(dst, &v, 4);
  }
}

/* Evaluate all tags at one logical index. When `points` is non-null the s-th
 * store writes element `pi` of points[s] instead of its view. */
static void eval_one(const orc_command* c, const int* cls, uint32_t* val,
                     const int64_t* idx, void* const* points, int64_t pi) {
  int s = 0;
  for (int t = 0; t < c->n_ops; ++t) {
    const orc_op* op = &c->ops[t];
    switch (op->kind) {
      case ORC_LOAD_TENSOR:
        val[t] = load_elem(op, view_offset(op, idx, c->rank));
        break;
      case ORC_LOAD_SCALAR:
        val[t] = op->scalar_bits;
        break;
      case ORC_ADD:
        val[t] = cls[t] == CLS_INT ? orc_iadd(val[op->a], val[op->b])
                                   : orc_fadd(val[op->a], val[op->b]);
        break;
      case ORC_SUB:
        val[t] = cls[t] == CLS_INT ? orc_isub(val[op->a], val[op->b])
                                   : orc_fsub(val[op->a], val[op->b]);
        break;
      case ORC_MUL:
        val[t] = cls[t] == CLS_INT ? orc_imul(val[op->a], val[op->b])
                                   : orc_fmul(val[op->a], val[op->b]);
        break;
      case ORC_NEG:
        val[t] = cls[t] == CLS_INT ? orc_ineg(val[op->a]) : orc_fneg(val[op->a]);
        break;
      case ORC_DIV:
        val[t] = cls[t] == CLS_INT ? orc_idiv(val[op->a], val[op->b])
                                   : orc_fdiv(val[op->a], val[op->b]);
        break;
      case ORC_MIN:
        val[t] = cls[t] == CLS_INT ? orc_imin(val[op->a], val[op->b])
                                   : orc_fmin(val[op->a], val[op->b]);
        break;
      case ORC_MAX:
        val[t] = cls[t] == CLS_INT ? orc_imax(val[op->a], val[op->b])
                                   : orc_fmax(val[op->a], val[op->b]);
        break;
      case ORC_ABS:
        val[t] = cls[t] == CLS_INT ? orc_iabs(val[op->a]) : orc_fabs(val[op->a]);
        break;
      case ORC_TO_F32:
        val[t] = cls[op->a] == CLS_INT ? orc_i2f(val[op->a]) : val[op->a];
        break;
      case ORC_TO_I32:
        val[t] = cls[op->a] == CLS_INT ? val[op->a] : orc_f2i(val[op->a]);
        break;
      case ORC_LT:
      case ORC_LE:
      case ORC_GT:
      case ORC_GE:
      case ORC_EQ:
      case ORC_NE:
      case ORC_ULT:
      case ORC_ULE:
      case ORC_UGT:
      case ORC_UGE:
        val[t] = orc_compare(op->kind, cls[op->a] == CLS_INT, val[op->a], val[op->b]);
        break;
      case ORC_SELECT:
        val[t] = val[op->c] != 0u ? val[op->a] : val[op->b];
        break;
      case ORC_STORE: {
        if (op->dtype == ORC_B1) {
          uint32_t bit = val[op->a] != 0u;
          if (points) {
            ((uint8_t*)points[s])[pi] = (uint8_t)bit;
          } else {
            int64_t off = view_offset(op, idx, c->rank);
            char* wp = (char*)op->ptr + (off / 32) * 4;
            uint32_t w;
            memcpy(&w, wp, 4);
            w = (w & ~(1u << (off % 32))) | (bit << (off % 32));
            memcpy(wp, &w, 4);
          }
          ++s;
          break;
        }
        size_t es = elem_size(op->dtype);
        char* dst;
        if (points) {
          dst = (char*)points[s] + pi * (int64_t)es;
        } else {
          dst = (char*)op->ptr + view_offset(op, idx, c->rank) * (int64_t)es;
        }
        convert_store(op->dtype, val[op->a], dst);
        ++s;
        break;
      }
    }
  }
}

/* Row-major logical multi-index of a linear index (Flatten's order). */
static void unflatten(const orc_command* c, int64_t lin, int64_t* idx) {
  for (int k = c->rank - 1; k >= 0; --k) {
    idx[k] = lin % c->sizes[k];
    lin /= c->sizes[k];
  }
}

static int64_t total_elems(const orc_command* c) {
  int64_t n = 1;
  for (int k = 0; k < c->rank; ++k) n *= c->sizes[k];
  return n;
}

/* The view's strides are the row-major strides of the logical sizes. */
static int dense_row_major(const orc_command* c, const orc_op* op) {
  int64_t acc = 1;
  for (int k = c->rank - 1; k >= 0; --k) {
    if (c->sizes[k] != 1 && op->strides[k] != acc) return 0;
    acc *= c->sizes[k];
  }
  return 1;
}

static int check_command(const orc_command* c) {
  if (!c || c->n_ops < 0 || (c->n_ops > 0 && !c->ops)) return ORC_EBAD;
  if (c->rank < 0 || c->rank > ORC_MAX_RANK) return ORC_EBAD;
  for (int k = 0; k < c->rank; ++k)
    if (c->sizes[k] < 0) return ORC_EBAD;
  return ORC_OK;
}

int orc_eval_range(const orc_command* c, int64_t begin, int64_t end) {
  int rc = check_command(c);
  if (rc) return rc;
  int64_t n = total_elems(c);
  if (begin < 0) begin = 0;
  if (end > n) end = n;
  if (begin >= end || c->n_ops == 0) return ORC_OK;
  int* cls = (int*)malloc(sizeof(int) * (size_t)c->n_ops);
  uint32_t* val = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)c->n_ops);
  if (!cls || !val) {
    free(cls);
    free(val);
    return ORC_ENOMEM;
  }
  rc = classify(c, cls);
  if (rc == ORC_OK) {
    int64_t idx[ORC_MAX_RANK] = {0, 0, 0, 0};
    for (int64_t e = begin; e < end; ++e) {
      unflatten(c, e, idx);
      eval_one(c, cls, val, idx, NULL, 0);
    }
    /* B1 stores over dense row-major views: once the last element is
     * written, the bits of its word past it are 0 */
    if (end == n && n % 32 != 0) {
      for (int t = 0; t < c->n_ops; ++t) {
        const orc_op* op = &c->ops[t];
        if (op->kind != ORC_STORE || op->dtype != ORC_B1 || !dense_row_major(c, op)) continue;
        char* wp = (char*)op->ptr + ((n - 1) / 32) * 4;
        uint32_t w;
        memcpy(&w, wp, 4);
        w &= (1u << (n % 32)) - 1u;
        memcpy(wp, &w, 4);
      }
    }
  }
  free(cls);
  free(val);
  return rc;
}

int orc_eval_points(const orc_command* c, const int64_t* lin, int64_t n,
                    void* const* store_out) {
  int rc = check_command(c);
  if (rc) return rc;
  if (n <= 0 || c->n_ops == 0) return ORC_OK;
  if (!lin || !store_out) return ORC_EBAD;
  int64_t total = total_elems(c);
  int* cls = (int*)malloc(sizeof(int) * (size_t)c->n_ops);
  uint32_t* val = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)c->n_ops);
  if (!cls || !val) {
    free(cls);
    free(val);
    return ORC_ENOMEM;
  }
  rc = classify(c, cls);
  if (rc == ORC_OK) {
    int64_t idx[ORC_MAX_RANK] = {0, 0, 0, 0};
    for (int64_t i = 0; i < n; ++i) {
      if (lin[i] < 0 || lin[i] >= total) {
        rc = ORC_EBAD;
        break;
      }
      unflatten(c, lin[i], idx);
      eval_one(c, cls, val, idx, store_out, i);
    }
  }
  free(cls);
  free(val);
  return rc;
}
