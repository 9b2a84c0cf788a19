/*
 * cmd.h - fused tensor Command execution on one GPU (GB300, sm_103a): C ABI.
 *
 * A Command is built up from operations, each of which creates a tag that
 * later operations refer to (rocRoller, "Design Overview", section "Command
 * Class"). The operations here are the ones that section and section
 * "Operations" describe: loading a tensor or a scalar, a T_Execute block of
 * E_ operations applied elementwise to vectors or scalars, and storing a
 * tensor. Load and store operations take their data as runtime arguments
 * supplied at launch (section "CommandArgument"): a device pointer with the
 * tensor's sizes and strides, or a scalar value. Tensor indexing follows the
 * coordinate-transform reading of section "Kernel Graph": a tensor element
 * at logical multi-index (i_0, ..., i_{r-1}) lives at element offset
 * sum_k i_k * stride_k, and logical elements are ordered row-major (the
 * Flatten transform).
 *
 * cmd_compile lowers a Command to a compact register-slot program (dead-tag
 * elimination, common-subexpression reuse, slot allocation by liveness) held
 * in GPU constant memory; cmd_launch runs it as one fused pass over the
 * tensors (section "Command Kernel": a compiled Command is launched many
 * times with different runtime arguments).
 *
 * Arithmetic. Float Commands compute in binary32 with one round-to-nearest-
 * even rounding per E op and no fused multiply-add; denormals are kept.
 * binary16 and bfloat16 loads widen exactly; stores to them round once, to
 * nearest even (overflow to infinity). int32 Commands wrap modulo 2^32.
 * E_Neg flips the sign bit of a float and is 0 - x for an int.
 *
 * Ownership. The library owns Command and kernel objects (create/destroy
 * pairs below). The caller owns every device buffer and stream; buffers must
 * stay valid until the launched work has completed on its stream. Scalar
 * values are copied at launch.
 *
 * Errors. Every call returns a cmd_status; CMD_OK is 0. A failing call leaves
 * its object unchanged and records a message for cmd_last_error() (per
 * thread). Nothing is thrown across this interface. A launch is asynchronous:
 * cmd_launch reports launch-phase errors and cmd_sync_status reports the
 * completion phase.
 *
 * Threading. A Command or kernel object may be used by one thread at a time;
 * distinct objects may be used concurrently.
 */
#ifndef CMD_H
#define CMD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CMD_ABI_VERSION 3

/* limits */
#define CMD_MAX_RANK 4      /* logical dims of a tensor view */
#define CMD_MAX_TAGS 128    /* operations (tags) in one Command */
#define CMD_MAX_LOADS 16    /* live Load_Tensor ops after dead-tag elimination */
#define CMD_MAX_STORES 8    /* Store_Tensor ops */
#define CMD_MAX_SCALARS 16  /* live Load_Scalar ops */
#define CMD_MAX_SLOTS 32    /* simultaneously live values in the lowered program */
#define CMD_MAX_KERNELS 48  /* compiled kernels alive at once, per device */

typedef enum cmd_status {
  CMD_OK = 0,
  CMD_ERR_NULL = 1,           /* a required pointer argument is NULL */
  CMD_ERR_BAD_TAG = 2,        /* a tag does not name a usable earlier result */
  CMD_ERR_TYPE = 3,           /* int/float mix, or a dtype not allowed here */
  CMD_ERR_SHAPE = 4,          /* rank, size or stride mismatch / out of range */
  CMD_ERR_ALIAS = 5,          /* a store overlaps another tensor argument */
  CMD_ERR_ALIGN = 6,          /* a pointer is not aligned to its element size */
  CMD_ERR_STATE = 7,          /* wrong object state (e.g. wrong device) */
  CMD_ERR_LIMIT = 8,          /* a CMD_MAX_* limit would be exceeded */
  CMD_ERR_CUDA = 9,           /* the CUDA runtime reported an error */
  CMD_ERR_DEVICE_TIMEOUT = 10,/* a device-side wait gave up */
  CMD_ERR_NOMEM = 11,         /* host allocation failed */
  CMD_ERR_ARG = 12            /* runtime arguments missing, repeated or unknown */
} cmd_status;

/* Element types. CMD_B1 is a store type only: one bit per element, packed
 * into little-endian 32-bit words (element at bit offset k of the view goes
 * to bit k % 32 of word k / 32); its view must be dense row-major (the bit
 * offset of an element is its row-major logical index), the buffer 4-byte
 * aligned and ceil(numel / 32) words long. Each word is written whole: the
 * bits of the last word past the last element are 0. The packed prediction
 * store of the Silk page's threshold classification ("AMDGPU Backend",
 * section "Code Object Format") is this store of a comparison result. */
typedef enum cmd_dtype { CMD_F32 = 0, CMD_F16 = 1, CMD_BF16 = 2, CMD_I32 = 3, CMD_B1 = 4 } cmd_dtype;

/* Elementwise operations of a T_Execute block (rocRoller, "Design Overview",
 * section "Operations": E_ operations such as Add and Subtract on vectors or
 * scalars; DIV .. TO_I32 follow the operations an Expression supports,
 * section "Expression", whose special cases the pages leave open and which
 * are fixed here). Float ops round once to nearest even; int ops wrap modulo
 * 2^32.
 *   ADD, SUB, MUL, NEG  as their names say; NEG flips a float's sign bit.
 *   DIV     float: IEEE division. int: truncates toward zero; x / 0 = -1 and
 *           INT_MIN / -1 = INT_MIN (so that every input has one result).
 *   MIN/MAX float: IEEE 754-2019 minimumNumber / maximumNumber (a NaN loses to
 *           a number; -0 is less than +0). int: signed.
 *   ABS     float: sign bit cleared. int: |x| modulo 2^32 (|INT_MIN| = INT_MIN).
 *   TO_F32  int -> float, rounded to nearest even; a float is unchanged.
 *   TO_I32  float -> int, truncated toward zero and saturated to the int32
 *           range, NaN -> 0; an int is unchanged.
 *   LT, LE, GT, GE, EQ, NE  the int 1 when a (rel) b holds, else 0: IEEE
 *           comparisons for floats (a NaN operand makes all but NE false;
 *           -0 == +0), signed for ints.
 *   ULT, ULE, UGT, UGE      ints compared as unsigned 32-bit numbers (the
 *           unsigned threshold comparison of the Silk page's threshold
 *           classification, "AMDGPU Backend", section "Code Object Format").
 *   SELECT  a if the int c is nonzero, else b; a and b of one class.
 * NEG, ABS, TO_F32 and TO_I32 take one operand (b is ignored); only SELECT
 * reads c. */
typedef enum cmd_eop {
  CMD_E_ADD = 0,
  CMD_E_SUB = 1,
  CMD_E_MUL = 2,
  CMD_E_NEG = 3,
  CMD_E_DIV = 4,
  CMD_E_MIN = 5,
  CMD_E_MAX = 6,
  CMD_E_ABS = 7,
  CMD_E_TO_F32 = 8,
  CMD_E_TO_I32 = 9,
  CMD_E_LT = 10,
  CMD_E_LE = 11,
  CMD_E_GT = 12,
  CMD_E_GE = 13,
  CMD_E_EQ = 14,
  CMD_E_NE = 15,
  CMD_E_ULT = 16,
  CMD_E_ULE = 17,
  CMD_E_UGT = 18,
  CMD_E_UGE = 19,
  CMD_E_SELECT = 20
} cmd_eop;

typedef int32_t cmd_tag;
typedef struct cmd_command* cmd_command_t;
typedef struct cmd_kernel* cmd_kernel_t;

/* Operand of an E op inside the same cmd_add_execute call: the result of the
 * block's i-th op (i smaller than the referring op's index). */
#define CMD_LOCAL(i) ((cmd_tag)(-1 - (i)))

/* One E op: result = a (op) b, op(a) for the one-operand ops (b ignored), or
 * c ? a : b for SELECT (c ignored by every other op). a, b and c are tags of
 * earlier Load_Tensor, Load_Scalar or E results, or CMD_LOCAL(i). */
typedef struct cmd_xop {
  int32_t op; /* cmd_eop */
  cmd_tag a;
  cmd_tag b;
  cmd_tag c;
} cmd_xop;

/* Runtime argument of a Load_Tensor or Store_Tensor tag: a pointer the GPU
 * can address and the view. sizes are the logical sizes (equal for every
 * tensor of the Command); strides are in elements, >= 0, one per logical dim.
 * The pointer is device memory, or pinned (page-locked) host memory from
 * cudaHostAlloc / cudaHostRegister, whose address is valid on the device
 * under unified addressing: the kernel then reads and writes it across the
 * host link itself, with no separate copy (on a Grace host, the coherent
 * CPU-GPU link). Pageable host memory is not accepted by this contract. */
typedef struct cmd_tensor_arg {
  cmd_tag tag;
  int32_t rank;
  void* ptr;
  int64_t sizes[CMD_MAX_RANK];
  int64_t strides[CMD_MAX_RANK];
} cmd_tensor_arg;

/* Runtime argument of a Load_Scalar tag. Use .f32 for a CMD_F32 scalar and
 * .i32 for a CMD_I32 scalar. */
typedef struct cmd_scalar_arg {
  cmd_tag tag;
  union {
    float f32;
    int32_t i32;
    uint32_t bits;
  } v;
} cmd_scalar_arg;

typedef struct cmd_runtime_args {
  const cmd_tensor_arg* tensors;
  int32_t n_tensors;
  const cmd_scalar_arg* scalars;
  int32_t n_scalars;
} cmd_runtime_args;

/* Result of lowering, for inspection (cmd_lower / cmd_kernel_info). */
typedef struct cmd_program_info {
  int32_t n_live_ops;   /* E ops left after dead-tag elimination and reuse */
  int32_t n_loads;      /* live Load_Tensor ops (each read once per element) */
  int32_t n_scalars;    /* live Load_Scalar ops */
  int32_t n_stores;
  int32_t n_slots;      /* register slots the program needs */
  int32_t n_words;      /* program words, including the end marker */
  int32_t tier;         /* executor family: 0 = 2 slots, 1 = 4, 2 = 8, 3 = 32, 4 = 16 */
  int32_t n_moves;      /* copies the two-address form needed */
  int32_t extended;     /* 1 if the program has a live division, comparison or
                           select, or a packed-bit store: it runs the
                           executors' extended variant; 0: the base variant,
                           whose loop carries none of that code */
} cmd_program_info;

/* Which executor a launch would use (cmd_plan_launch). */
typedef enum cmd_path {
  CMD_PATH_NONE = 0,    /* nothing to do (no elements or no stores) */
  CMD_PATH_CONTIG = 1,  /* every view dense row-major and aligned, or all off the vector
                           alignment by one number of elements (the few elements before
                           they align run per element): vector loads/stores. 1-D views
                           whose loads sit off the stores' alignment by other numbers of
                           elements also take it, up to 16 live values (shifted loads;
                           the first 4 to 7 and the last 4 or more elements run per
                           element). With
                           merged_rank 2: rows, every view unit-stride along the columns,
                           each row starting on a 4-element boundary (a load's row stride
                           may be 0) and a whole number of warp chunks long (padded or
                           sliced row-major tensors); or rows at offsets from that
                           boundary with row strides of whole 4-element vectors, whose
                           first and last few columns run per element */
  CMD_PATH_TILE2D = 2,  /* 2-D views, row-direct or transposed, staged through shared memory */
  CMD_PATH_GENERIC = 3  /* any other sizes/strides: per-element offsets */
} cmd_path;

typedef struct cmd_launch_plan {
  int32_t path;           /* cmd_path */
  int32_t merged_rank;    /* rank after dropping size-1 dims and merging dims */
  int64_t merged_sizes[CMD_MAX_RANK];
  int64_t n_elements;     /* logical elements */
  int64_t bytes;          /* live loads read once + stores written once */
  int32_t n_transposed;   /* loads staged through shared memory (tile path) */
  /* How a CMD_PATH_CONTIG launch splits (all 0 otherwise): the contiguous
   * kernel runs contig_elements elements (of every row, for a row walk)
   * starting head_elements in; the elements before and after them run per
   * element. shifted_loads counts the loads read shifted (at another offset
   * from the vector alignment than the stores). */
  int64_t head_elements;
  int64_t contig_elements;
  int32_t shifted_loads;
} cmd_launch_plan;

int32_t cmd_abi_version(void);
const char* cmd_status_string(cmd_status s);
/* Message of the last failing call on this thread ("" if none). */
const char* cmd_last_error(void);

/* ---- building a Command (host only) -------------------------------------- */

/* Create an empty Command; *out receives the handle. */
cmd_status cmd_create(cmd_command_t* out);
/* Destroy a Command (NULL is ignored). Compiled kernels stay valid. */
void cmd_destroy(cmd_command_t cmd);

/* Tag the next operation added to cmd will receive. */
cmd_status cmd_next_tag(cmd_command_t cmd, cmd_tag* out);

/* Load_Tensor of element type dtype and logical rank 0..CMD_MAX_RANK. */
cmd_status cmd_add_load_tensor(cmd_command_t cmd, cmd_dtype dtype, int32_t rank, cmd_tag* out);

/* Load_Scalar of type CMD_F32 or CMD_I32 (broadcast to every element). */
cmd_status cmd_add_load_scalar(cmd_command_t cmd, cmd_dtype dtype, cmd_tag* out);

/* One T_Execute block of n E ops (1..CMD_MAX_TAGS). Op i receives tag
 * first + i, written to out_tags[i] when out_tags is non-NULL. Operands of a
 * two-operand op must both be float-valued or both int-valued (ULT .. UGE:
 * int-valued); comparisons make int values, TO_F32 a float value and TO_I32
 * an int value; SELECT's c must be int-valued and its a and b of one class.
 * On error nothing is added. */
cmd_status cmd_add_execute(cmd_command_t cmd, const cmd_xop* ops, int32_t n, cmd_tag* out_tags);

/* Store_Tensor of tag src as element type dtype, logical rank `rank`. A float
 * value may be stored as CMD_F32, CMD_F16 or CMD_BF16; an int value as
 * CMD_I32 or CMD_B1 (the bit is value != 0). */
cmd_status cmd_add_store(cmd_command_t cmd, cmd_tag src, cmd_dtype dtype, int32_t rank, cmd_tag* out);

/* ---- text form -------------------------------------------------------- */

/* A Command as text and back (rocRoller, "Design Overview", section
 * "Serialization": a Command converts to and from YAML, for saving, caching
 * and inspecting kernel definitions). The text is a small fixed subset of
 * YAML that cmd_to_yaml writes and cmd_from_yaml reads:
 *
 *   # comments (from a '#' at a line's start or after a space) and blank lines
 *   version: 1
 *   operations:
 *     - {kind: load_tensor, tag: 0, dtype: f32, rank: 1}
 *     - {kind: load_scalar, tag: 1, dtype: f32}
 *     - kind: execute                       (one T_Execute block)
 *       ops:
 *         - {tag: 2, op: mul, a: 0, b: 1}
 *         - {tag: 3, op: neg, a: 2}         (one-operand ops: a only)
 *         - {tag: 4, op: select, a: 2, b: 3, c: 5}
 *     - {kind: store_tensor, tag: 5, src: 4, dtype: f32, rank: 1}
 *
 * Keys of a {...} mapping may come in any order; tags must be 0, 1, 2, ...
 * in order (they are the tags the Command gets), operands refer to earlier
 * tags, op names are those of cmd_eop in lower case (add .. uge, select) and
 * dtype names f32, f16, bf16, i32, b1. The reader rebuilds the Command
 * through cmd_create and the cmd_add_* calls, so it applies all of their
 * checks; the same Command lowers to the same program. */

/* Write cmd's text form into buf (NUL-terminated, truncated to size);
 * *needed receives the full length + 1 when non-NULL. */
cmd_status cmd_to_yaml(cmd_command_t cmd, char* buf, int64_t size, int64_t* needed);

/* Build a new Command from len bytes of text form (len < 0: text is
 * NUL-terminated). On success *out owns it (release with cmd_destroy); on
 * error nothing is allocated, CMD_ERR_ARG (or the failing builder call's
 * status) is returned and cmd_last_error() names the line. */
cmd_status cmd_from_yaml(const char* text, int64_t len, cmd_command_t* out);

/* ---- lowering ---------------------------------------------------------- */

/* Lower cmd on the host only (no GPU needed): fills *info and, when words is
 * non-NULL, up to cap program words. For inspection and tests. */
cmd_status cmd_lower(cmd_command_t cmd, cmd_program_info* info, uint32_t* words, int32_t cap);

/* Lower cmd and place the program in constant memory of the current CUDA
 * device. Synchronises that device (it may reuse the constant slot of a
 * destroyed kernel), so do not call it during stream capture. Allocates the
 * kernel's 256-byte device error word (cudaMalloc) and waits until it is
 * cleared. The Command may be destroyed afterwards. All tensors of the
 * Command must share one rank. */
cmd_status cmd_compile(cmd_command_t cmd, cmd_kernel_t* out);

/* Like cmd_compile, but allocates no device memory. For callers that cannot
 * call cudaMalloc: programs whose device memory belongs wholly to their own
 * pool or to a framework's allocator (a fixed arena sized at start-up, a
 * budget that the CUDA allocator must not grow), where an allocation outside
 * the pool is refused or breaks the accounting. The only device memory a
 * kernel needs beyond its inputs and outputs is one 4-byte error word for the
 * tile executor's bounded waits; kernels from this call keep it in a static
 * 256-byte array of the library (one word per constant-memory program slot,
 * so at most CMD_MAX_KERNELS such words) that every GPU which loads the
 * library holds until the process exits. Like cmd_compile, the call uploads
 * the program with synchronous copies, clears the word and waits for the
 * clear, and synchronises the device when it reuses a program slot: make it
 * outside any stream capture. The first call on a device also looks up the
 * array's device address on that device. The word then keeps whatever the
 * kernel's launches report until cmd_sync_status reads and clears it, and
 * launches of the same kernel that overlap on the GPU share (race on) it.
 * Launch, inspect and destroy the kernel with the usual calls; none of them
 * allocates device memory for such a kernel. The pages have no counterpart
 * of this entry point. */
cmd_status cmd_compile_static_scratch(cmd_command_t cmd, cmd_kernel_t* out);

/* Lower cmd into a kernel handle without touching any GPU. Such a kernel can
 * be inspected (cmd_kernel_info, cmd_kernel_dump) and planned
 * (cmd_plan_launch) but not launched (CMD_ERR_STATE). */
cmd_status cmd_lower_kernel(cmd_command_t cmd, cmd_kernel_t* out);

/* Release a kernel and its constant-memory slot (NULL is ignored). Work
 * already launched with it must not still be pending. */
void cmd_kernel_destroy(cmd_kernel_t k);

cmd_status cmd_kernel_info(cmd_kernel_t k, cmd_program_info* info);

/* Text listing of the lowered program into buf (NUL-terminated, truncated to
 * size); *needed receives the full length + 1 when non-NULL. */
cmd_status cmd_kernel_dump(cmd_kernel_t k, char* buf, int64_t size, int64_t* needed);

/* ---- launching --------------------------------------------------------- */

/* Validate args against the kernel and report the executor it would use,
 * without touching the GPU (and so without looking at where the memory lies:
 * cmd_launch runs a CMD_PATH_TILE2D plan on the generic executor when a load
 * is not in device memory). */
cmd_status cmd_plan_launch(cmd_kernel_t k, const cmd_runtime_args* args, cmd_launch_plan* plan);

/* Validate args and enqueue one fused pass on stream cuda_stream (a
 * cudaStream_t; NULL = the legacy default stream), on the device the kernel
 * was compiled for, which must be current. Every live Load_Tensor, Store_Tensor
 * and Load_Scalar tag needs exactly one argument; arguments for dead tags may
 * be omitted. Stores must not overlap any other tensor argument (an identical
 * view of the same element type, used in place, is allowed) and must not
 * overlap themselves. Tensors may lie in pinned host memory (see
 * cmd_tensor_arg); views that would take the tile executor run on the
 * generic one whenever a load lies anywhere but in device memory, since the
 * tile executor's TMA copies are issued on device memory only. Returns after the launch is enqueued (asynchronous). A
 * launch with zero elements does nothing. Safe to capture in a CUDA graph. */
cmd_status cmd_launch(cmd_kernel_t k, const cmd_runtime_args* args, void* cuda_stream);

/* Wait for cuda_stream and report the completion phase of work launched on
 * it with k: CMD_OK; CMD_ERR_CUDA with the runtime's message; or
 * CMD_ERR_DEVICE_TIMEOUT when a device-side wait of the tile executor (an
 * mbarrier wait on its shared-memory pipeline) ran past the time limit and
 * the kernel stopped instead of hanging. The kernel's device error word is
 * cleared when it is reported, on cuda_stream, and the call waits for the
 * clear; a launch of k on another stream that runs meanwhile may have its
 * report cleared with it. */
cmd_status cmd_sync_status(cmd_kernel_t k, void* cuda_stream);

/* Process-wide settings of the device-side waits: the time limit of every
 * bounded wait (default 2 s), and a test hook: with force_timeout != 0 the
 * tile executor's consumer warps wait on a barrier that nothing completes, so
 * the timeout path runs (the launch then writes no output and
 * cmd_sync_status returns CMD_ERR_DEVICE_TIMEOUT). */
cmd_status cmd_configure_waits(uint64_t timeout_ns, int32_t force_timeout);

/* ---- diagnostics --------------------------------------------------------- */

/* Device allocations (cudaMalloc calls that succeeded) this library has made
 * in this process, on every device together: one per kernel from cmd_compile
 * and none from any other call. For tests and for callers that account for
 * device memory. */
int64_t cmd_device_allocations(void);

#ifdef __cplusplus
}
#endif

#endif /* CMD_H */
