/*
 * cmd_oracle.h - plain, slow CPU oracle for fused Command execution.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference legs may load or call this library.
 * The product (the CUDA executor and its C ABI) never links, imports or calls
 * it, and it shares no code, header, table or helper with the product.
 *
 * What it computes (rocRoller, "Design Overview"):
 *   - a Command is a list of operations; adding one creates a tag and later
 *     operations refer to earlier results by tag (section "Command Class");
 *   - Load and Store operations carry runtime arguments: a pointer plus the
 *     size/stride description of the tensor, or a scalar value (sections
 *     "Operations" and "CommandArgument");
 *   - a T_Execute block holds E_ operations applied elementwise to vectors
 *     or scalars (section "Operations");
 *   - tensor indexes come from sizes and strides; the logical element order
 *     is row-major, as the Flatten coordinate transform makes it (section
 *     "Kernel Graph").
 *
 * The oracle evaluates, for every logical index in row-major order, every tag
 * in creation order, with no dead-tag elimination, no common-subexpression
 * reuse and no reordering: the Command exactly as written.
 *
 * Arithmetic readings (the pages leave these open; see the design notes):
 *   - float E ops: one round-to-nearest-even rounding to binary32 per op, the
 *     operands exactly as written, no fused multiply-add. Computed here as the
 *     binary64 result rounded once more to binary32; for + - x with
 *     53 >= 2*24 + 2 that second rounding is innocuous (S. A. Figueroa,
 *     "When is double rounding innocuous?", SIGNUM Newsletter 1995).
 *   - denormals are kept (no flush to zero) on input and output;
 *   - int32 E ops: two's-complement arithmetic modulo 2^32;
 *   - E_Neg flips the sign bit of a float and is 0 - x for an int;
 *   - half and bfloat16 inputs widen exactly to binary32; stores round once,
 *     to nearest even, overflow to infinity; NaN payloads are not pinned.
 *   - E_Div: binary32 division rounded once to nearest even (IEEE 754 6.3 /
 *     7.3 for zeros and infinities); int32 division truncates toward zero,
 *     x / 0 = -1 and INT_MIN / -1 = INT_MIN (the convention the RISC-V ISA
 *     manual fixes for its DIV instruction, taken here so that every input
 *     has one result).
 *   - E_Min / E_Max: IEEE 754-2019 minimumNumber / maximumNumber: a NaN
 *     operand loses to a number, and -0 counts as less than +0; int32 signed.
 *   - E_Abs: the sign bit cleared for a float; |x| modulo 2^32 for an int
 *     (|INT_MIN| = INT_MIN).
 *   - E_ToF32: an int converts with one round to nearest even; a float is
 *     unchanged. E_ToI32: a float truncates toward zero and saturates to the
 *     int32 range, NaN gives 0; an int is unchanged.
 *   - comparisons (LT, LE, GT, GE, EQ, NE) give the int 1 when they hold and
 *     0 otherwise: IEEE 754 comparisons for floats (any NaN operand makes all
 *     of them false except NE, which is true; -0 equals +0), signed for
 *     ints; ULT, ULE, UGT, UGE compare ints as unsigned 32-bit numbers (the
 *     Silk page's threshold classification: an unsigned threshold
 *     comparison of a loaded u32, "AMDGPU Backend", section "Code Object
 *     Format").
 *   - SELECT(c, a, b) is a when the int c is nonzero, else b (a and b of one
 *     class).
 *   - a B1 store packs one bit per element, (value != 0), at bit offset
 *     sum(index * stride) of the buffer taken as little-endian u32 words
 *     (bit k of word k / 32); for a dense row-major view the bits of the
 *     last word past the last element are 0.
 */
#ifndef CMD_ORACLE_H
#define CMD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_I32 = 3, ORC_B1 = 4 /* store only */ };

/* operation kinds */
enum {
  ORC_LOAD_TENSOR = 0,
  ORC_LOAD_SCALAR = 1,
  ORC_ADD = 2,
  ORC_SUB = 3,
  ORC_MUL = 4,
  ORC_NEG = 5,
  ORC_STORE = 6,
  ORC_DIV = 7,
  ORC_MIN = 8,
  ORC_MAX = 9,
  ORC_ABS = 10,
  ORC_TO_F32 = 11,
  ORC_TO_I32 = 12,
  ORC_LT = 13,
  ORC_LE = 14,
  ORC_GT = 15,
  ORC_GE = 16,
  ORC_EQ = 17,
  ORC_NE = 18,
  ORC_ULT = 19,
  ORC_ULE = 20,
  ORC_UGT = 21,
  ORC_UGE = 22,
  ORC_SELECT = 23
};

/* status codes */
enum { ORC_OK = 0, ORC_EBAD = -1, ORC_ETYPE = -2, ORC_ENOMEM = -3 };

#define ORC_MAX_RANK 4

/* One operation; its tag is its index in the command's op array. */
typedef struct {
  int32_t kind;      /* ORC_LOAD_TENSOR ... ORC_STORE */
  int32_t dtype;     /* element type of a tensor load/store, or of a scalar */
  int32_t a;         /* first operand tag (E ops); source tag (STORE) */
  int32_t b;         /* second operand tag (two-operand ops, SELECT) */
  int32_t c;         /* SELECT: the condition's tag */
  void* ptr;         /* LOAD_TENSOR / STORE: host base address */
  int64_t strides[ORC_MAX_RANK]; /* LOAD_TENSOR / STORE: stride per logical dim, in elements */
  uint32_t scalar_bits;          /* LOAD_SCALAR: the value's bits (binary32 or int32) */
} orc_op;

typedef struct {
  int32_t n_ops;
  const orc_op* ops;
  int32_t rank;                  /* 0..4; every tensor shares these logical sizes */
  int64_t sizes[ORC_MAX_RANK];
} orc_command;

/* Evaluate logical (row-major) indices [begin, end) and write every store to
 * its view. Returns ORC_OK or a negative status (invalid command). */
int orc_eval_range(const orc_command* cmd, int64_t begin, int64_t end);

/* Evaluate the n logical indices lin[0..n) and, instead of writing the views,
 * put the value of the s-th STORE op (in tag order) at element i of
 * store_out[s], in that store's element type (one byte, 0 or 1, for B1). */
int orc_eval_points(const orc_command* cmd, const int64_t* lin, int64_t n,
                    void* const* store_out);

/* Per-op arithmetic and conversions, exposed so tests can pin them. */
uint32_t orc_fadd(uint32_t x, uint32_t y);
uint32_t orc_fsub(uint32_t x, uint32_t y);
uint32_t orc_fmul(uint32_t x, uint32_t y);
uint32_t orc_fneg(uint32_t x);
uint32_t orc_iadd(uint32_t x, uint32_t y);
uint32_t orc_isub(uint32_t x, uint32_t y);
uint32_t orc_imul(uint32_t x, uint32_t y);
uint32_t orc_ineg(uint32_t x);
uint32_t orc_fdiv(uint32_t x, uint32_t y);
uint32_t orc_idiv(uint32_t x, uint32_t y);
uint32_t orc_fmin(uint32_t x, uint32_t y);
uint32_t orc_fmax(uint32_t x, uint32_t y);
uint32_t orc_imin(uint32_t x, uint32_t y);
uint32_t orc_imax(uint32_t x, uint32_t y);
uint32_t orc_fabs(uint32_t x);
uint32_t orc_iabs(uint32_t x);
uint32_t orc_i2f(uint32_t x);
uint32_t orc_f2i(uint32_t x);
/* kind: ORC_LT .. ORC_UGE; is_int selects the int (or unsigned) comparison. */
uint32_t orc_compare(int32_t kind, int32_t is_int, uint32_t x, uint32_t y);
uint16_t orc_f32_to_f16(uint32_t x);
uint16_t orc_f32_to_bf16(uint32_t x);
uint32_t orc_f16_to_f32(uint16_t h);
uint32_t orc_bf16_to_f32(uint16_t h);

/* Bulk forms of the four conversions, for exhaustive pins over bit ranges. */
void orc_f32_to_f16_n(const uint32_t* x, uint16_t* out, int64_t n);
void orc_f32_to_bf16_n(const uint32_t* x, uint16_t* out, int64_t n);

#ifdef __cplusplus
}
#endif

#endif /* CMD_ORACLE_H */
