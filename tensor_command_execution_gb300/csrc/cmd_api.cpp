// cmd_api.cpp - the C ABI of cmd.h: Command building, lowering to the
// register-slot program, launch validation and executor selection.
//
// Lowering follows the rocRoller "Design Overview" pipeline in spirit
// (sections "Kernel Graph", "Expression", "Registers", "Command Kernel"): the
// Command's tag graph is rewritten (dead tags dropped, identical operations
// reused), values are given registers by their lifetimes, and a compact
// program is emitted for the hand-written executors to run.
#include "../../include/cmd.h"

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <tuple>
#include <vector>

#include "cmd_internal.h"

namespace {

thread_local std::string g_last_error;

cmd_status fail(cmd_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

enum OpKind { kLoad = 0, kScalar = 1, kExec = 2, kStore = 3 };
enum ValClass { kFloat = 0, kInt = 1, kNone = 2 };

struct Op {
  int kind;
  int dtype;  // load/store element type, scalar type
  int rank;   // load/store logical rank
  int eop;    // kExec: cmd_eop
  int a, b;   // kExec operands (b = -1 for one-operand ops); kStore: a = source
  int c;      // SELECT: the condition (else -1)
  int cls;    // value class of the result
  int block = -1;  // kExec: which T_Execute block (cmd_add_execute call) it came in
};

const char* dtype_name(int dt) {
  switch (dt) {
    case CMD_F32: return "f32";
    case CMD_F16: return "f16";
    case CMD_BF16: return "bf16";
    case CMD_I32: return "i32";
    case CMD_B1: return "b1";
  }
  return "?";
}

int elem_size(int dt) { return (dt == CMD_F16 || dt == CMD_BF16) ? 2 : 4; }

// The text form's names of the E ops, in cmd_eop order.
const char* const kEopNames[] = {"add", "sub", "mul", "neg", "div", "min", "max", "abs", "to_f32", "to_i32", "lt",
                                 "le", "gt", "ge", "eq", "ne", "ult", "ule", "ugt", "uge", "select"};
const char* eop_name(int eop) { return eop >= 0 && eop <= CMD_E_SELECT ? kEopNames[eop] : "?"; }

// E ops that take one operand.
bool is_unary(int eop) { return eop == CMD_E_NEG || eop == CMD_E_ABS || eop == CMD_E_TO_F32 || eop == CMD_E_TO_I32; }
bool is_compare(int eop) { return eop >= CMD_E_LT && eop <= CMD_E_UGE; }
// E ops whose two operands commute exactly (IEEE 754 and modulo 2^32).
bool is_commutative(int eop) {
  return eop == CMD_E_ADD || eop == CMD_E_MUL || eop == CMD_E_MIN || eop == CMD_E_MAX || eop == CMD_E_EQ ||
         eop == CMD_E_NE;
}

// Element types of loads (and of scalars: f32/i32 only, checked apart).
bool valid_dtype(int dt) { return dt >= CMD_F32 && dt <= CMD_I32; }
bool valid_store_dtype(int dt) { return dt >= CMD_F32 && dt <= CMD_B1; }

// One instruction of the two-address program, before encoding. kSlotX
// stands for the staging slot (the tier's last slot), fixed at encoding.
constexpr int kSlotX = -2;
struct Instr {
  enum Kind { kBin, kUn, kBinS, kMovS, kSt, kCmpX, kCmpS, kSel, kSelS, kSDiv } kind;
  int op;   // BinOp / UnOp / StoreType / CmpOp
  int d;    // destination slot (kSlotX: the staging slot)
  int s;    // source slot
  int aux;  // scalar index or output index
};

struct Program {
  std::vector<int> load_tags;    // slot j holds the j-th live load
  std::vector<int> scalar_tags;  // scalar index k
  std::vector<int> store_tags;   // output index o
  std::vector<Instr> code;
  std::vector<uint32_t> words;
  int n_live_e = 0;
  int n_slots = 0;
  int n_moves = 0;
  int tier = cmdx::kTier4;
  bool extended = false;  // uses an extended op or store: runs the executors' extended variant
  bool uses_x = false;   // comparisons or selects read the staging slot
  // scalars derived at launch (after the program's own): {DerivedKind, own scalar index}
  std::vector<std::pair<int, int>> derived;
};

}  // namespace

namespace cmdx {
// Record msg for cmd_last_error() and return s (for the host sources that
// build Commands through the public API, e.g. the text-form reader).
cmd_status host_fail(cmd_status s, const std::string& msg) { return fail(s, msg); }
}  // namespace cmdx

struct cmd_command {
  std::vector<Op> ops;
  int n_blocks = 0;  // T_Execute blocks added so far
};

struct cmd_kernel {
  std::vector<Op> ops;
  Program prog;
  int rank = 0;
  int device = -1;
  int slot = -1;
  uint32_t* err = nullptr;  // device error word of the tile executor's bounded waits
  bool err_owned = true;    // false when err points into static device memory
};

namespace {

// ---- device-side wait limit and the test hook that forces a timeout ----------
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int32_t> g_force_timeout{0};
// successful device allocations made by this library (cmd_device_allocations)
std::atomic<int64_t> g_device_allocs{0};

// Zero n bytes of device memory at p on the legacy default stream and wait
// until that is done: a plain cudaMemset of device memory may return before
// it completes, and a launch on a non-blocking stream made right after would
// not be ordered after it (its report could then be erased).
cudaError_t clear_device_now(void* p, size_t n) {
  cudaError_t e = cudaMemsetAsync(p, 0, n, cudaStreamLegacy);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cudaStreamLegacy);
  return e;
}

// ---- constant-memory program slots, per device -----------------------------
std::mutex g_slot_mu;
std::map<int, std::vector<int>> g_slot_state;  // 0 never used, 1 in use, 2 freed

int acquire_slot(int device, bool* reused) {
  std::lock_guard<std::mutex> g(g_slot_mu);
  auto& st = g_slot_state[device];
  if (st.empty()) st.assign(cmdx::kMaxPrograms, 0);
  for (int pass = 0; pass < 2; ++pass) {
    for (int i = 0; i < cmdx::kMaxPrograms; ++i) {
      if ((pass == 0 && st[i] == 0) || (pass == 1 && st[i] == 2)) {
        *reused = st[i] == 2;
        st[i] = 1;
        return i;
      }
    }
  }
  return -1;
}

void release_slot(int device, int slot) {
  std::lock_guard<std::mutex> g(g_slot_mu);
  auto it = g_slot_state.find(device);
  if (it != g_slot_state.end() && slot >= 0 && slot < (int)it->second.size()) it->second[slot] = 2;
}

// ---- lowering --------------------------------------------------------------

cmd_status check_command(const cmd_command* c, int* rank_out) {
  int rank = -1;
  bool any_store = false;
  for (size_t t = 0; t < c->ops.size(); ++t) {
    const Op& op = c->ops[t];
    if (op.kind == kLoad || op.kind == kStore) {
      if (rank < 0) rank = op.rank;
      if (op.rank != rank)
        return fail(CMD_ERR_SHAPE, "tag " + std::to_string(t) + " has rank " + std::to_string(op.rank) +
                                       " but an earlier tensor has rank " + std::to_string(rank) +
                                       "; every tensor of a Command shares the logical sizes");
    }
    if (op.kind == kStore) any_store = true;
  }
  (void)any_store;
  *rank_out = rank < 0 ? 0 : rank;
  return CMD_OK;
}

cmd_status lower(const std::vector<Op>& ops, Program* P) {
  const int n = (int)ops.size();
  // common-subexpression reuse: an E op with the same (op, operands) as an
  // earlier one takes that one's value; Add and Mul are commutative exactly
  // (bit for bit in IEEE 754 and modulo 2^32), so their operands are ordered.
  std::vector<int> rep(n);
  std::map<std::tuple<int, int, int, int>, int> seen;
  for (int t = 0; t < n; ++t) {
    const Op& op = ops[t];
    rep[t] = t;
    if (op.kind != kExec) continue;
    int a = rep[op.a];
    int b = is_unary(op.eop) ? -1 : rep[op.b];
    int c = op.eop == CMD_E_SELECT ? rep[op.c] : -1;
    if (is_commutative(op.eop) && b < a) std::swap(a, b);
    auto key = std::make_tuple(op.eop, a, b, c);
    auto it = seen.find(key);
    if (it != seen.end())
      rep[t] = it->second;
    else
      seen.emplace(key, t);
  }
  // dead-tag elimination: keep what a store reaches
  std::vector<char> live(n, 0);
  for (int t = n - 1; t >= 0; --t) {
    const Op& op = ops[t];
    if (op.kind == kStore) {
      live[t] = 1;
      live[rep[op.a]] = 1;
    } else if (op.kind == kExec && live[t] && rep[t] == t) {
      live[rep[op.a]] = 1;
      if (!is_unary(op.eop)) live[rep[op.b]] = 1;
      if (op.eop == CMD_E_SELECT) live[rep[op.c]] = 1;
    }
  }
  std::vector<int> slot_of(n, -1), sidx(n, -1);
  P->load_tags.clear();
  P->scalar_tags.clear();
  P->store_tags.clear();
  P->code.clear();
  P->n_live_e = 0;
  P->n_moves = 0;
  for (int t = 0; t < n; ++t) {
    if (!live[t]) continue;
    if (ops[t].kind == kLoad) {
      slot_of[t] = (int)P->load_tags.size();
      P->load_tags.push_back(t);
    } else if (ops[t].kind == kScalar) {
      sidx[t] = (int)P->scalar_tags.size();
      P->scalar_tags.push_back(t);
    } else if (ops[t].kind == kStore) {
      P->store_tags.push_back(t);
    } else if (rep[t] == t) {
      ++P->n_live_e;
    }
  }
  if ((int)P->load_tags.size() > cmdx::kMaxLoads)
    return fail(CMD_ERR_LIMIT, "more than " + std::to_string(cmdx::kMaxLoads) + " live Load_Tensor ops");
  if ((int)P->store_tags.size() > cmdx::kMaxStores)
    return fail(CMD_ERR_LIMIT, "more than " + std::to_string(cmdx::kMaxStores) + " Store_Tensor ops");
  if ((int)P->scalar_tags.size() > cmdx::kMaxScalars)
    return fail(CMD_ERR_LIMIT, "more than " + std::to_string(cmdx::kMaxScalars) + " live Load_Scalar ops");

  // emission order: stores of loaded or scalar values first, then each live
  // E op in tag order followed by the stores of its value
  struct Event { bool store; int tag; };
  std::vector<Event> ev;
  for (int t : P->store_tags) {
    int src = rep[ops[t].a];
    if (ops[src].kind != kExec) ev.push_back({true, t});
  }
  std::vector<std::vector<int>> stores_of(n);
  for (int t : P->store_tags) {
    int src = rep[ops[t].a];
    if (ops[src].kind == kExec) stores_of[src].push_back(t);
  }
  for (int t = 0; t < n; ++t) {
    if (ops[t].kind != kExec || !live[t] || rep[t] != t) continue;
    ev.push_back({false, t});
    for (int s : stores_of[t]) ev.push_back({true, s});
  }
  std::vector<int> last_use(n, -1);
  for (int i = 0; i < (int)ev.size(); ++i) {
    const Op& op = ops[ev[i].tag];
    if (ev[i].store) {
      last_use[rep[op.a]] = i;
    } else {
      last_use[rep[op.a]] = i;
      if (!is_unary(op.eop)) last_use[rep[op.b]] = i;
      if (op.eop == CMD_E_SELECT) last_use[rep[op.c]] = i;
    }
  }
  // slots
  bool busy[cmdx::kMaxSlots + 1] = {};
  int in_use = 0, peak = 0;
  int n_loads = (int)P->load_tags.size();
  for (int j = 0; j < n_loads; ++j) busy[j] = true;
  in_use = peak = n_loads;
  bool overflow = false;
  auto alloc = [&]() -> int {
    for (int i = 0; i < cmdx::kMaxSlots; ++i) {
      if (!busy[i]) {
        busy[i] = true;
        ++in_use;
        peak = std::max(peak, in_use);
        return i;
      }
    }
    overflow = true;
    return cmdx::kMaxSlots;  // never encoded: lowering fails below
  };
  auto release = [&](int s) {
    if (s >= 0 && s < cmdx::kMaxSlots && busy[s]) {
      busy[s] = false;
      --in_use;
    }
  };
  auto is_scalar = [&](int t) { return ops[t].kind == kScalar; };
  auto emit = [&](Instr::Kind k, int op, int d, int s, int aux) { P->code.push_back({k, op, d, s, aux}); };
  auto store_type = [&](int dt) { return dt; /* cmd_dtype numbering matches StoreType */ };
  std::map<std::pair<int, int>, int> sdiv_base;  // (float/int, own scalar) -> first derived index
  P->derived.clear();

  for (int i = 0; i < (int)ev.size(); ++i) {
    const int t = ev[i].tag;
    const Op& op = ops[t];
    if (ev[i].store) {
      int src = rep[op.a];
      int o = (int)(std::find(P->store_tags.begin(), P->store_tags.end(), t) - P->store_tags.begin());
      if (is_scalar(src)) {
        int d = alloc();
        emit(Instr::kMovS, cmdx::kMov, d, 0, sidx[src]);
        emit(Instr::kSt, store_type(op.dtype), 0, d, o);
        release(d);
      } else {
        emit(Instr::kSt, store_type(op.dtype), 0, slot_of[src], o);
        if (last_use[src] == i) release(slot_of[src]);
      }
      continue;
    }
    const bool ints = op.cls == kInt;
    const int a = rep[op.a];
    if (is_unary(op.eop)) {
      const bool a_int = ops[a].cls == kInt;
      int uop;
      if (op.eop == CMD_E_NEG) uop = ints ? cmdx::kINeg : cmdx::kFNeg;
      else if (op.eop == CMD_E_ABS) uop = ints ? cmdx::kIAbs : cmdx::kFAbs;
      else if (op.eop == CMD_E_TO_F32) uop = a_int ? cmdx::kI2F : cmdx::kMov;
      else uop = a_int ? cmdx::kMov : cmdx::kF2I;
      int d;
      if (is_scalar(a)) {
        d = alloc();
        emit(Instr::kMovS, cmdx::kMov, d, 0, sidx[a]);
        if (uop != cmdx::kMov) emit(Instr::kUn, uop, d, d, 0);
      } else if (last_use[a] == i) {
        d = slot_of[a];
        if (uop != cmdx::kMov) emit(Instr::kUn, uop, d, d, 0);
      } else {
        d = alloc();
        emit(Instr::kUn, uop, d, slot_of[a], 0);
      }
      slot_of[t] = d;
      continue;
    }
    const int b = rep[op.b];
    if (is_compare(op.eop) || op.eop == CMD_E_SELECT) {
      // both read the staging slot X, filled right before them
      const bool sa = is_scalar(a), sb = is_scalar(b);
      const bool die_a = !sa && last_use[a] == i;
      const bool die_b = !sb && last_use[b] == i;
      auto to_x = [&](int x) {  // X = value of tag x
        P->uses_x = true;
        ++P->n_moves;
        if (is_scalar(x)) emit(Instr::kMovS, cmdx::kMov, kSlotX, 0, sidx[x]);
        else emit(Instr::kUn, cmdx::kMov, kSlotX, slot_of[x], 0);
      };
      auto copy_into_new = [&](int x) {  // a fresh slot holding the value of tag x
        int d = alloc();
        ++P->n_moves;
        if (is_scalar(x)) emit(Instr::kMovS, cmdx::kMov, d, 0, sidx[x]);
        else emit(Instr::kUn, cmdx::kMov, d, slot_of[x], 0);
        return d;
      };
      int d;
      if (is_compare(op.eop)) {
        const bool f = ops[a].cls == kFloat;
        // CmpOp groups list LT LE GT GE EQ NE in cmd_eop order
        int cop = op.eop >= CMD_E_ULT ? cmdx::kCULt + (op.eop - CMD_E_ULT)
                                      : (f ? cmdx::kCFLt : cmdx::kCILt) + (op.eop - CMD_E_LT);
        if (sb) {  // d = a rel scalar b
          d = die_a ? slot_of[a] : copy_into_new(a);
          emit(Instr::kCmpS, cop, d, 0, sidx[b]);
        } else if (sa) {  // d = b (swapped rel) scalar a
          d = die_b ? slot_of[b] : copy_into_new(b);
          emit(Instr::kCmpS, cmdx::cmp_swap(cop), d, 0, sidx[a]);
        } else if (die_a) {
          to_x(b);
          d = slot_of[a];
          emit(Instr::kCmpX, cop, d, 0, 0);
          if (die_b && b != a) release(slot_of[b]);
        } else if (die_b) {
          to_x(a);
          d = slot_of[b];
          emit(Instr::kCmpX, cmdx::cmp_swap(cop), d, 0, 0);
        } else {
          d = copy_into_new(a);
          to_x(b);
          emit(Instr::kCmpX, cop, d, 0, 0);
        }
      } else {
        const int c = rep[op.c];
        to_x(c);
        // d holds a (the value when c != 0), then takes b where c == 0
        if (die_a) d = slot_of[a];
        else d = copy_into_new(a);
        if (sb) emit(Instr::kSelS, 0, d, 0, sidx[b]);
        else emit(Instr::kSel, 0, d, slot_of[b], 0);
        // operands whose last use this is and whose slot d did not take
        int dying[2] = {b, c};
        for (int k = 0; k < 2; ++k) {
          const int x = dying[k];
          if (is_scalar(x) || last_use[x] != i || slot_of[x] == d) continue;
          if (k == 1 && x == b) continue;  // released already as b
          release(slot_of[x]);
        }
      }
      slot_of[t] = d;
      continue;
    }
    int bop, rsub;  // rsub: the reversed form, d = x (op) d
    switch (op.eop) {
      case CMD_E_ADD: bop = rsub = ints ? cmdx::kIAdd : cmdx::kFAdd; break;
      case CMD_E_SUB:
        bop = ints ? cmdx::kISub : cmdx::kFSub;
        rsub = ints ? cmdx::kIRsub : cmdx::kFRsub;
        break;
      case CMD_E_MUL: bop = rsub = ints ? cmdx::kIMul : cmdx::kFMul; break;
      case CMD_E_DIV:
        bop = ints ? cmdx::kIDiv : cmdx::kFDiv;
        rsub = ints ? cmdx::kIRdiv : cmdx::kFRdiv;
        break;
      case CMD_E_MIN: bop = rsub = ints ? cmdx::kIMin : cmdx::kFMin; break;
      default: bop = rsub = ints ? cmdx::kIMax : cmdx::kFMax; break;
    }
    const bool commut = is_commutative(op.eop);
    const bool sa = is_scalar(a), sb = is_scalar(b);
    const bool die_a = !sa && last_use[a] == i;
    const bool die_b = !sb && last_use[b] == i;
    if (op.eop == CMD_E_DIV && !sa && sb) {
      // a tensor value divided by a scalar: through constants the host
      // derives from the scalar at launch (a reciprocal, or a multiply-high
      // constant and shift), when the scalar table has room for them
      const int o = ints ? 1 : 0;
      const auto key = std::make_pair(o, sidx[b]);
      auto it = sdiv_base.find(key);
      int base = it != sdiv_base.end() ? it->second : -1;
      const int need = o == 0 ? 2 : 3;
      if (base < 0 && (int)(P->scalar_tags.size() + P->derived.size()) + need <= cmdx::kMaxScalars) {
        base = (int)(P->scalar_tags.size() + P->derived.size());
        P->derived.push_back({cmdx::kDerCopy, sidx[b]});
        if (o == 0) {
          P->derived.push_back({cmdx::kDerRecip, sidx[b]});
        } else {
          P->derived.push_back({cmdx::kDerIMagic, sidx[b]});
          P->derived.push_back({cmdx::kDerIShift, sidx[b]});
        }
        sdiv_base[key] = base;
      }
      if (base >= 0) {
        int d;
        if (die_a) {
          d = slot_of[a];
        } else {
          d = alloc();
          ++P->n_moves;
          emit(Instr::kUn, cmdx::kMov, d, slot_of[a], 0);
        }
        emit(Instr::kSDiv, o, d, 0, base);
        slot_of[t] = d;
        continue;
      }
    }
    auto src = [&](int bo, int d, int x) {  // d = d (bo) x
      if (is_scalar(x)) emit(Instr::kBinS, bo, d, 0, sidx[x]);
      else emit(Instr::kBin, bo, d, slot_of[x], 0);
    };
    int d;
    if (die_a) {
      d = slot_of[a];
      src(bop, d, b);
      if (die_b && b != a) release(slot_of[b]);
    } else if (die_b) {
      d = slot_of[b];
      src(commut ? bop : rsub, d, a);
    } else {
      d = alloc();
      ++P->n_moves;
      if (sa && sb) {
        emit(Instr::kMovS, cmdx::kMov, d, 0, sidx[a]);
        src(bop, d, b);
      } else if (sa) {
        emit(Instr::kUn, cmdx::kMov, d, slot_of[b], 0);
        src(commut ? bop : rsub, d, a);
      } else {
        emit(Instr::kUn, cmdx::kMov, d, slot_of[a], 0);
        src(bop, d, b);
      }
    }
    slot_of[t] = d;
  }
  if (overflow || peak > cmdx::kMaxSlots)
    return fail(CMD_ERR_LIMIT, "the program needs more than " + std::to_string(cmdx::kMaxSlots) +
                                   " simultaneously live values");
  // a program that uses the staging slot needs one slot above its values
  P->n_slots = std::max(peak, 1) + (P->uses_x ? 1 : 0);
  if (P->n_slots > cmdx::kMaxSlots)
    return fail(CMD_ERR_LIMIT, "the program needs more than " + std::to_string(cmdx::kMaxSlots - 1) +
                                   " simultaneously live values besides the staging slot of its comparisons");
  P->tier = P->n_slots <= 2    ? cmdx::kTier2
            : P->n_slots <= 4  ? cmdx::kTier4
            : P->n_slots <= 8  ? cmdx::kTier8
            : P->n_slots <= 16 ? cmdx::kTier16
                               : cmdx::kTier32;

  // encode
  P->words.clear();
  // the extended variant: division, comparisons, select, packed-bit stores
  P->extended = false;
  for (const Instr& in : P->code) {
    const bool div = ((in.kind == Instr::kBin || in.kind == Instr::kBinS) && in.op >= cmdx::kFDiv && in.op <= cmdx::kIRdiv) ||
                     in.kind == Instr::kSDiv;
    const bool cmp_sel = in.kind == Instr::kCmpX || in.kind == Instr::kCmpS || in.kind == Instr::kSel ||
                         in.kind == Instr::kSelS;
    const bool bits = in.kind == Instr::kSt && in.op == cmdx::kStB1;
    if (div || cmp_sel || bits) P->extended = true;
  }
  const int S = cmdx::tier_slots(P->tier);
  const int X = S - 1;  // the staging slot
  for (Instr& in : P->code)
    if (in.d == kSlotX) in.d = X;
  // an op that reads the staging slot never writes it or reads it as its
  // other operand: the executors have no case for that
  for (const Instr& in : P->code) {
    const bool reads_x = in.kind == Instr::kCmpX || in.kind == Instr::kSel || in.kind == Instr::kSelS;
    if (reads_x && (in.d == X || (in.kind == Instr::kSel && in.s == X)))
      return fail(CMD_ERR_STATE, "internal: the lowering placed a value in the staging slot");
  }
  for (const Instr& in : P->code) {
    uint32_t w = 0;
    if (!cmdx::tier_wide(P->tier)) {
      switch (in.kind) {
        case Instr::kBin: w = cmdx::fz_bin(S, in.op, in.d, in.s); break;
        case Instr::kUn: w = cmdx::fz_un(S, in.op, in.d, in.s); break;
        case Instr::kBinS: w = cmdx::fz_bin_scalar(S, in.op, in.d) | uint32_t(in.aux) << 16; break;
        case Instr::kMovS: w = cmdx::fz_movs(S, in.d) | uint32_t(in.aux) << 16; break;
        case Instr::kSt: w = cmdx::fz_store(S, in.op, in.s) | uint32_t(in.aux) << 16; break;
        case Instr::kCmpX: w = cmdx::fz_cmpx(S, in.op, in.d); break;
        case Instr::kCmpS: w = cmdx::fz_cmps(S, in.op, in.d) | uint32_t(in.aux) << 16; break;
        case Instr::kSel: w = cmdx::fz_sel(S, in.d, in.s); break;
        case Instr::kSelS: w = cmdx::fz_sels(S, in.d) | uint32_t(in.aux) << 16; break;
        case Instr::kSDiv: w = cmdx::fz_sdiv(S, in.op, in.d) | uint32_t(in.aux) << 16; break;
      }
    } else {
      switch (in.kind) {
        case Instr::kBin: w = cmdx::wd_word(cmdx::kWBin0 + in.op, in.d, in.s, 0); break;
        case Instr::kUn: w = cmdx::wd_word(cmdx::kWUn0 + in.op, in.d, in.s, 0); break;
        case Instr::kCmpX: w = cmdx::wd_word(cmdx::kWCmp0 + in.op, in.d, X, 0); break;
        case Instr::kCmpS: w = cmdx::wd_word((cmdx::kWCmp0 + in.op) | cmdx::kWScalar, in.d, 0, in.aux); break;
        case Instr::kSel: w = cmdx::wd_word(cmdx::kWSel, in.d, in.s, 0); break;
        case Instr::kSelS: w = cmdx::wd_word(cmdx::kWSel | cmdx::kWScalar, in.d, 0, in.aux); break;
        case Instr::kSDiv: w = cmdx::wd_word(cmdx::kWSDiv0 + in.op, in.d, 0, in.aux); break;
        case Instr::kBinS: w = cmdx::wd_word((cmdx::kWBin0 + in.op) | cmdx::kWScalar, in.d, 0, in.aux); break;
        case Instr::kMovS: w = cmdx::wd_word((cmdx::kWUn0 + cmdx::kMov) | cmdx::kWScalar, in.d, 0, in.aux); break;
        case Instr::kSt: w = cmdx::wd_word(cmdx::kWStore0 + in.op, 0, in.s, in.aux); break;
      }
    }
    P->words.push_back(w);
  }
  P->words.push_back(!cmdx::tier_wide(P->tier) ? cmdx::fz_end(S) : cmdx::wd_word(cmdx::kWEnd, 0, 0, 0));
  if ((int)P->words.size() > cmdx::kMaxProgramWords)
    return fail(CMD_ERR_LIMIT, "the lowered program has " + std::to_string(P->words.size()) +
                                   " words; the limit is " + std::to_string(cmdx::kMaxProgramWords));
  return CMD_OK;
}

void fill_info(const Program& P, cmd_program_info* info) {
  info->n_live_ops = P.n_live_e;
  info->n_loads = (int32_t)P.load_tags.size();
  info->n_scalars = (int32_t)P.scalar_tags.size();
  info->n_stores = (int32_t)P.store_tags.size();
  info->n_slots = P.n_slots;
  info->n_words = (int32_t)P.words.size();
  info->tier = P.tier;
  info->n_moves = P.n_moves;
  info->extended = P.extended ? 1 : 0;
}

// ---- launch validation and planning ----------------------------------------

struct View {
  int tag;
  int dtype;
  void* ptr;
  int64_t st[cmdx::kMaxRank];
};

struct Plan {
  int path = CMD_PATH_NONE;
  int64_t n = 0;
  // contiguous path: elements before the first one at which every pointer is
  // aligned for the vector width (they run on the generic executor)
  int64_t head = 0;
  // contiguous path over rows (two merged dims, each view unit-stride along
  // the inner one): the row count; 0 for one dense range
  int64_t rows = 0;
  // contiguous path with loads off the stores' vector alignment (1-D): the
  // head then ends where the stores align, 4 elements further on
  bool shifted = false;
  int mrank = 0;
  int64_t msizes[cmdx::kMaxRank] = {1, 1, 1, 1};
  std::vector<View> loads, stores;       // in slot / output order
  int64_t ml[cmdx::kMaxLoads][cmdx::kMaxRank];    // merged strides of loads
  int64_t ms[cmdx::kMaxStores][cmdx::kMaxRank];   // merged strides of stores
  uint32_t scal[cmdx::kMaxScalars] = {};
  int n_trans = 0;
  int64_t bytes = 0;
  // tile executor: merged-dim indices of the tile's row and column dims and
  // of the (up to two) batch dims, outer first
  int tile_row = -1, tile_col = -1, n_batch = 0, batch[2] = {-1, -1};
};

// A scalar derived at launch from the program's scalar v (see DerivedKind).
uint32_t derive_scalar(int kind, uint32_t v) {
  if (kind == cmdx::kDerCopy) return v;
  if (kind == cmdx::kDerRecip) {
    // RN(1/s): the binary64 quotient rounded once more to binary32 (innocuous,
    // 53 >= 2*24 + 2); 0 (no fast path) outside [2^-60, 2^60] or for 0, inf, NaN
    float s;
    std::memcpy(&s, &v, 4);
    const double a = std::fabs((double)s);
    if (!(a >= std::ldexp(1.0, -60) && a <= std::ldexp(1.0, 60))) return 0u;
    const float r = (float)(1.0 / (double)s);
    uint32_t rb;
    std::memcpy(&rb, &r, 4);
    return rb;
  }
  // int32 division by d, truncating (Granlund and Montgomery, "Division by
  // invariant integers using multiplication", PLDI 1994, section 5):
  // l = max(ceil(log2 |d|), 1), m = 1 + floor(2^(31 + l) / |d|) - 2^32,
  // shift l - 1; d = 0 and d = -1 take the general division
  const int32_t d = (int32_t)v;
  if (d == 0 || d == -1) return kind == cmdx::kDerIMagic ? 0u : cmdx::kSDivSlow;
  const uint64_t ad = d < 0 ? (uint64_t)(-(int64_t)d) : (uint64_t)d;
  int l = 0;
  while ((uint64_t(1) << l) < ad) ++l;
  if (l < 1) l = 1;
  if (kind == cmdx::kDerIShift) return (uint32_t)(l - 1);
  const int64_t m = 1 + (int64_t)((uint64_t(1) << (31 + l)) / ad) - (int64_t(1) << 32);
  return (uint32_t)(int32_t)m;
}

// Largest element offset reached by a view (+1), over dims of size > 1.
int64_t view_extent(const int64_t* sizes, const int64_t* st, int rank) {
  int64_t e = 0;
  for (int k = 0; k < rank; ++k)
    if (sizes[k] > 1) e += (sizes[k] - 1) * st[k];
  return e + 1;
}

// Sufficient condition for a view to address distinct elements: with dims of
// size > 1 sorted by stride, each stride exceeds the span of the smaller ones.
bool view_injective(const int64_t* sizes, const int64_t* st, int rank) {
  std::vector<std::pair<int64_t, int64_t>> d;
  for (int k = 0; k < rank; ++k)
    if (sizes[k] > 1) d.push_back({st[k], sizes[k]});
  std::sort(d.begin(), d.end());
  int64_t span = 0;  // largest offset reachable by the smaller dims
  for (auto& x : d) {
    if (x.first <= span) return false;
    span += (x.second - 1) * x.first;
  }
  return true;
}

cmd_status plan_launch(const cmd_kernel* k, const cmd_runtime_args* args, Plan* pl) {
  const auto& ops = k->ops;
  const int n = (int)ops.size();
  const int rank = k->rank;
  if (!args) return fail(CMD_ERR_NULL, "args is NULL");
  if (args->n_tensors < 0 || args->n_scalars < 0) return fail(CMD_ERR_ARG, "negative argument count");
  if (args->n_tensors > 0 && !args->tensors) return fail(CMD_ERR_NULL, "args->tensors is NULL");
  if (args->n_scalars > 0 && !args->scalars) return fail(CMD_ERR_NULL, "args->scalars is NULL");
  std::vector<int> targ(n, -1), sarg(n, -1);
  int64_t sizes[cmdx::kMaxRank] = {1, 1, 1, 1};
  bool have_sizes = false;
  for (int i = 0; i < args->n_tensors; ++i) {
    const cmd_tensor_arg& a = args->tensors[i];
    if (a.tag < 0 || a.tag >= n || (ops[a.tag].kind != kLoad && ops[a.tag].kind != kStore))
      return fail(CMD_ERR_BAD_TAG, "tensor argument " + std::to_string(i) + " names tag " + std::to_string(a.tag) +
                                       ", which is not a Load_Tensor or Store_Tensor of this kernel");
    if (targ[a.tag] >= 0) return fail(CMD_ERR_ARG, "tag " + std::to_string(a.tag) + " has two tensor arguments");
    targ[a.tag] = i;
    if (a.rank != rank)
      return fail(CMD_ERR_SHAPE, "tensor argument for tag " + std::to_string(a.tag) + " has rank " +
                                     std::to_string(a.rank) + ", the Command's tensors have rank " + std::to_string(rank));
    for (int d = 0; d < rank; ++d) {
      if (a.sizes[d] < 0) return fail(CMD_ERR_SHAPE, "negative size for tag " + std::to_string(a.tag));
      if (a.strides[d] < 0)
        return fail(CMD_ERR_SHAPE, "negative stride for tag " + std::to_string(a.tag) + " (strides must be >= 0)");
    }
    if (!have_sizes) {
      for (int d = 0; d < rank; ++d) sizes[cmdx::kMaxRank - rank + d] = a.sizes[d];
      have_sizes = true;
    } else {
      for (int d = 0; d < rank; ++d)
        if (sizes[cmdx::kMaxRank - rank + d] != a.sizes[d])
          return fail(CMD_ERR_SHAPE, "tag " + std::to_string(a.tag) + " has logical size " + std::to_string(a.sizes[d]) +
                                         " in dim " + std::to_string(d) + ", another tensor has " +
                                         std::to_string(sizes[cmdx::kMaxRank - rank + d]));
    }
  }
  for (int i = 0; i < args->n_scalars; ++i) {
    const cmd_scalar_arg& a = args->scalars[i];
    if (a.tag < 0 || a.tag >= n || ops[a.tag].kind != kScalar)
      return fail(CMD_ERR_BAD_TAG, "scalar argument " + std::to_string(i) + " names tag " + std::to_string(a.tag) +
                                       ", which is not a Load_Scalar of this kernel");
    if (sarg[a.tag] >= 0) return fail(CMD_ERR_ARG, "tag " + std::to_string(a.tag) + " has two scalar arguments");
    sarg[a.tag] = i;
  }
  const Program& P = k->prog;
  for (int t : P.load_tags)
    if (targ[t] < 0) return fail(CMD_ERR_ARG, "no tensor argument for live Load_Tensor tag " + std::to_string(t));
  for (int t : P.store_tags)
    if (targ[t] < 0) return fail(CMD_ERR_ARG, "no tensor argument for Store_Tensor tag " + std::to_string(t));
  for (int t : P.scalar_tags)
    if (sarg[t] < 0) return fail(CMD_ERR_ARG, "no scalar argument for live Load_Scalar tag " + std::to_string(t));

  int64_t N = 1;
  for (int d = 0; d < cmdx::kMaxRank; ++d) N *= sizes[d];
  pl->n = N;
  pl->loads.clear();
  pl->stores.clear();
  auto mkview = [&](int t) {
    const cmd_tensor_arg& a = args->tensors[targ[t]];
    View v;
    v.tag = t;
    v.dtype = ops[t].dtype;
    v.ptr = a.ptr;
    for (int d = 0; d < cmdx::kMaxRank; ++d) v.st[d] = 0;
    for (int d = 0; d < rank; ++d) v.st[cmdx::kMaxRank - rank + d] = a.strides[d];
    return v;
  };
  for (int t : P.load_tags) pl->loads.push_back(mkview(t));
  for (int t : P.store_tags) pl->stores.push_back(mkview(t));
  for (size_t j = 0; j < P.scalar_tags.size(); ++j) pl->scal[j] = args->scalars[sarg[P.scalar_tags[j]]].v.bits;
  for (size_t j = 0; j < P.derived.size(); ++j)
    pl->scal[P.scalar_tags.size() + j] = derive_scalar(P.derived[j].first, pl->scal[P.derived[j].second]);
  pl->bytes = 0;
  for (auto& v : pl->loads) pl->bytes += N * elem_size(v.dtype);
  for (auto& v : pl->stores) pl->bytes += v.dtype == CMD_B1 ? (N + 31) / 32 * 4 : N * elem_size(v.dtype);
  if (N == 0 || P.store_tags.empty()) {
    pl->path = CMD_PATH_NONE;
    pl->mrank = 0;
    return CMD_OK;
  }
  // pointers
  auto check_ptr = [&](const View& v) -> cmd_status {
    if (!v.ptr) return fail(CMD_ERR_NULL, "NULL pointer for tag " + std::to_string(v.tag));
    if (reinterpret_cast<uintptr_t>(v.ptr) % (uintptr_t)elem_size(v.dtype))
      return fail(CMD_ERR_ALIGN, "pointer for tag " + std::to_string(v.tag) + " is not aligned to its " +
                                     std::to_string(elem_size(v.dtype)) + "-byte elements");
    return CMD_OK;
  };
  for (auto& v : pl->loads) if (cmd_status s = check_ptr(v)) return s;
  for (auto& v : pl->stores) if (cmd_status s = check_ptr(v)) return s;
  // packed-bit stores: the bit of an element is its row-major index, so the
  // view must be the dense row-major one
  bool any_b1 = false;
  for (auto& v : pl->stores) {
    if (v.dtype != CMD_B1) continue;
    any_b1 = true;
    int64_t acc = 1;
    for (int d = cmdx::kMaxRank - 1; d >= 0; --d) {
      if (sizes[d] != 1 && v.st[d] != acc)
        return fail(CMD_ERR_SHAPE, "the view of packed-bit Store_Tensor tag " + std::to_string(v.tag) +
                                       " is not dense row-major (bit i of the buffer is logical element i)");
      acc *= sizes[d];
    }
  }
  // bytes a view spans from its base
  auto span_bytes = [&](const View& v) -> int64_t {
    if (v.dtype == CMD_B1) return (N + 31) / 32 * 4;
    return view_extent(sizes, v.st, cmdx::kMaxRank) * elem_size(v.dtype);
  };
  // stores: injective, and not overlapping any other live tensor (an
  // identical view of the same element type read in place is allowed)
  for (size_t i = 0; i < pl->stores.size(); ++i) {
    const View& s = pl->stores[i];
    if (!view_injective(sizes, s.st, cmdx::kMaxRank))
      return fail(CMD_ERR_ALIAS, "the view of Store_Tensor tag " + std::to_string(s.tag) +
                                     " addresses some elements more than once");
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(s.ptr);
    const uintptr_t s1 = s0 + (uintptr_t)span_bytes(s);
    auto overlaps = [&](const View& o) {
      const uintptr_t o0 = reinterpret_cast<uintptr_t>(o.ptr);
      const uintptr_t o1 = o0 + (uintptr_t)span_bytes(o);
      return o0 < s1 && s0 < o1;
    };
    auto identical = [&](const View& o) {
      if (s.dtype == CMD_B1) return false;
      if (o.ptr != s.ptr || elem_size(o.dtype) != elem_size(s.dtype)) return false;
      for (int d = 0; d < cmdx::kMaxRank; ++d)
        if (sizes[d] > 1 && o.st[d] != s.st[d]) return false;
      return true;
    };
    for (size_t j = 0; j < pl->stores.size(); ++j)
      if (j != i && overlaps(pl->stores[j]))
        return fail(CMD_ERR_ALIAS, "Store_Tensor tags " + std::to_string(s.tag) + " and " +
                                       std::to_string(pl->stores[j].tag) + " overlap in memory");
    for (const View& l : pl->loads)
      if (overlaps(l) && !identical(l))
        return fail(CMD_ERR_ALIAS, "Store_Tensor tag " + std::to_string(s.tag) + " overlaps Load_Tensor tag " +
                                       std::to_string(l.tag) + " without being the identical view");
  }
  // merge dims: drop size-1 dims, then fuse neighbours that every view walks
  // as one (outer stride == inner stride * inner size)
  int64_t ms[cmdx::kMaxRank];
  int msrc[cmdx::kMaxRank];
  int m = 0;
  for (int d = 0; d < cmdx::kMaxRank; ++d)
    if (sizes[d] != 1) {
      ms[m] = sizes[d];
      msrc[m] = d;
      ++m;
    }
  std::vector<View*> all;
  for (auto& v : pl->loads) all.push_back(&v);
  for (auto& v : pl->stores) all.push_back(&v);
  // working strides per view over the kept dims
  std::vector<std::vector<int64_t>> wst(all.size());
  for (size_t i = 0; i < all.size(); ++i)
    for (int q = 0; q < m; ++q) wst[i].push_back(all[i]->st[msrc[q]]);
  for (int q = m - 2; q >= 0; --q) {
    bool ok = true;
    for (size_t i = 0; i < all.size() && ok; ++i) ok = wst[i][q] == wst[i][q + 1] * ms[q + 1];
    if (!ok) continue;
    ms[q] *= ms[q + 1];
    for (size_t i = 0; i < all.size(); ++i) {
      wst[i][q] = wst[i][q + 1];
      wst[i].erase(wst[i].begin() + q + 1);
    }
    for (int r = q + 1; r + 1 < m; ++r) ms[r] = ms[r + 1];
    --m;
  }
  pl->mrank = m;
  for (int d = 0; d < cmdx::kMaxRank; ++d) pl->msizes[d] = 1;
  for (int q = 0; q < m; ++q) pl->msizes[cmdx::kMaxRank - m + q] = ms[q];
  for (size_t j = 0; j < pl->loads.size(); ++j)
    for (int d = 0; d < cmdx::kMaxRank; ++d)
      pl->ml[j][d] = d < cmdx::kMaxRank - m ? 0 : wst[j][d - (cmdx::kMaxRank - m)];
  for (size_t j = 0; j < pl->stores.size(); ++j)
    for (int d = 0; d < cmdx::kMaxRank; ++d)
      pl->ms[j][d] = d < cmdx::kMaxRank - m ? 0 : wst[pl->loads.size() + j][d - (cmdx::kMaxRank - m)];

  auto aligned = [](const void* p, int bytes) { return reinterpret_cast<uintptr_t>(p) % (uintptr_t)bytes == 0; };
  // contiguous: one merged dim (or none) walked with stride 1 by every view,
  // and every pointer aligned for the vector width (4 elements per access)
  // (a packed-bit store writes single 32-bit words: 4-byte aligned suffices)
  bool contig = m <= 1;
  for (size_t i = 0; i < all.size() && contig; ++i) {
    if (m == 1 && wst[i][0] != 1) contig = false;
    const int vec = all[i]->dtype == CMD_B1 ? 4 : 4 * elem_size(all[i]->dtype);
    if (!aligned(all[i]->ptr, vec)) contig = false;
  }
  if (contig) {
    pl->path = CMD_PATH_CONTIG;
    return CMD_OK;
  }
  // One merged unit-stride dim whose pointers are all off the vector
  // alignment by the same number of elements (every tensor sliced at one
  // offset, say): after h = 4 - that number elements all of them are aligned,
  // so the first h run on the generic executor and the rest as above.
  // (Not with packed bits, whose words must start where the view does.)
  if (m <= 1 && !any_b1) {
    bool same = true;
    int64_t phase = -1;
    for (size_t i = 0; i < all.size() && same; ++i) {
      if (m == 1 && wst[i][0] != 1) same = false;
      const int64_t es = elem_size(all[i]->dtype);
      const int64_t ph = (int64_t)((reinterpret_cast<uintptr_t>(all[i]->ptr) / (uintptr_t)es) % 4);
      if (phase < 0) phase = ph;
      else if (ph != phase) same = false;
    }
    if (same && phase > 0 && pl->n > 4 - phase) {
      pl->path = CMD_PATH_CONTIG;
      pl->head = 4 - phase;
      return CMD_OK;
    }
  }
  // Shifted: one merged unit-stride dim whose stores all sit the same number
  // of elements off the vector alignment while some loads sit off it by
  // other numbers (x[1:] - x[:-1], say). The head runs up to where the
  // stores align, plus 4 elements; from there each load is read as aligned
  // vectors from up to 3 elements before it, each lane taking the end of its
  // elements from its right neighbour, and a tail of at least 4 elements is
  // left, so that those vectors stay inside the views. (Not in the 32-slot
  // tier, whose lanes hold groups of 2 elements, nor in the extended 8-slot
  // one, which is built with the dense-range kernel only; not with packed
  // bits.)
  const bool shift_tier = P.tier != cmdx::kTier32 && !(P.tier == cmdx::kTier8 && P.extended);
  if (m == 1 && !any_b1 && !pl->stores.empty() && shift_tier) {
    bool ok = true;
    int64_t sp = -1;
    for (size_t i = 0; i < all.size() && ok; ++i)
      if (wst[i][0] != 1) ok = false;
    for (const View& v : pl->stores) {
      const int64_t ph = (int64_t)((reinterpret_cast<uintptr_t>(v.ptr) / (uintptr_t)elem_size(v.dtype)) % 4);
      if (sp < 0) sp = ph;
      else if (ph != sp) ok = false;
    }
    const int64_t head = (4 - sp) % 4 + 4;
    const int64_t W = cmdx::contig_chunk(P.tier, P.extended, false);
    if (ok && pl->n >= head + W + 4) {
      pl->path = CMD_PATH_CONTIG;
      pl->head = head;
      pl->shifted = true;
      return CMD_OK;
    }
  }
  // Rows: two merged dims, every view unit-stride along the inner (column)
  // one, each row starting on the vector alignment (a base and a row stride
  // of whole 4-element vectors; a load's row stride may be 0, one row read
  // for every row), and rows a whole number of the contiguous executor's
  // warp chunks long, so that no chunk crosses a row: the contiguous kernel
  // then walks (row, chunk) pairs. Padded and sliced row-major tensors
  // (x[:, :n] of a wider x) take it. (Not with packed bits, nor in the
  // extended 8-slot tier, which is built with the dense-range kernel only.)
  const bool dense_only = P.tier == cmdx::kTier8 && P.extended;
  if (m == 2 && !any_b1 && !dense_only) {
    bool half2 = !pl->loads.empty();
    for (const auto& v : pl->loads) half2 = half2 && (v.dtype == CMD_F16 || v.dtype == CMD_BF16);
    const int64_t W = cmdx::contig_chunk(P.tier, P.extended, half2);
    bool rows_ok = ms[1] % W == 0 && ms[0] < (int64_t(1) << 30) && ms[1] / W < (int64_t(1) << 30);
    for (size_t i = 0; i < all.size() && rows_ok; ++i) {
      const int es = elem_size(all[i]->dtype);
      if (wst[i][1] != 1 || wst[i][0] % 4 != 0 || !aligned(all[i]->ptr, 4 * es)) rows_ok = false;
    }
    if (rows_ok) {
      pl->path = CMD_PATH_CONTIG;
      pl->rows = ms[0];
      return CMD_OK;
    }
  }
  // tile: two of the merged dims form the tile, the rest (at most two) are
  // batch dims. The column dim is the first store's unit-stride dim; the row
  // dim is the unit-stride dim of the loads that are not unit-stride along
  // the column dim (or, without such loads, the store's next smallest stride).
  // (not with packed-bit stores: those take the generic executor)
  if (m >= 2 && !cmdx::tier_wide(P.tier) && !pl->loads.empty() && !any_b1) {
    const size_t nl = pl->loads.size();
    int col = -1, row = -1;
    for (int q = 0; q < m; ++q)
      if (wst[nl][q] == 1) col = q;
    bool ok = col >= 0;
    for (size_t i = 0; i < nl && ok; ++i) {
      if (wst[i][col] == 1) continue;
      int unit = -1;
      for (int q = 0; q < m; ++q)
        if (q != col && wst[i][q] == 1) unit = q;
      if (unit < 0 || (row >= 0 && row != unit)) ok = false;
      else row = unit;
    }
    if (ok && row < 0) {
      for (int q = 0; q < m; ++q)
        if (q != col && (row < 0 || wst[nl][q] < wst[nl][row])) row = q;
    }
    int bd[2] = {-1, -1}, nbd = 0;
    for (int q = 0; q < m && ok; ++q)
      if (q != row && q != col) bd[nbd++] = q;
    int64_t tiles = 1;
    if (ok) {
      const int64_t R = ms[row], C = ms[col];
      tiles = ((R + cmdx::kTileRows - 1) / cmdx::kTileRows) * ((C + cmdx::kTileCols - 1) / cmdx::kTileCols);
      for (int b = 0; b < nbd; ++b) tiles *= ms[bd[b]];
      if (R >= (int64_t(1) << 31) || C >= (int64_t(1) << 31) || tiles >= (int64_t(1) << 31)) ok = false;
    }
    int n_trans = 0, stage = 0;
    for (size_t i = 0; i < all.size() && ok; ++i) {
      const bool is_store = i >= nl;
      const int es = elem_size(all[i]->dtype);
      const std::vector<int64_t>& v = wst[i];
      auto mul16 = [&](int64_t st) { return (st * es) % 16 == 0; };
      if (!aligned(all[i]->ptr, 16)) {
        ok = false;
        break;
      }
      for (int b = 0; b < nbd; ++b)
        if (!mul16(v[bd[b]])) ok = false;
      if (is_store) {
        // stores go out as 16-byte vectors along the column dim
        if (v[col] != 1 || !mul16(v[row])) ok = false;
        continue;
      }
      stage += cmdx::tile_stage_bytes(es);
      const bool trans = v[col] != 1;
      const int other = trans ? col : row;   // the load's non-unit tile dim
      if (v[other] != 0 && !mul16(v[other])) ok = false;
      if (trans) ++n_trans;
      // the load's TMA descriptor walks its dims with nonzero stride in
      // increasing stride order; each must step over the whole previous dim
      std::vector<std::pair<int64_t, int64_t>> d;  // (stride, size)
      d.push_back({1, ms[trans ? row : col]});
      if (v[other] != 0) d.push_back({v[other], ms[other]});
      for (int b = 0; b < nbd; ++b)
        if (v[bd[b]] != 0) d.push_back({v[bd[b]], ms[bd[b]]});
      std::sort(d.begin() + 1, d.end());
      for (size_t k2 = 1; k2 < d.size() && ok; ++k2)
        if (d[k2].first < d[k2 - 1].first * d[k2 - 1].second) ok = false;
    }
    if (ok && stage <= cmdx::kTileStageLimit) {
      pl->path = CMD_PATH_TILE2D;
      pl->n_trans = n_trans;
      pl->tile_row = row;
      pl->tile_col = col;
      pl->n_batch = nbd;
      pl->batch[0] = bd[0];
      pl->batch[1] = bd[1];
      return CMD_OK;
    }
  }
  // Shifted rows: rows as above, but starting at different offsets from the
  // vector alignment (x[:, 1:] of a wider x, say), views the tile executor
  // cannot take either (its copies start on 16-byte boundaries); every row stride
  // is a whole number of vectors, so each view keeps one offset on every
  // row. Per row, the columns up to where the stores align plus 4, and a
  // tail of at least 4, run per element; the columns between are whole warp
  // chunks on the contiguous kernel's row walk with shifted loads. Taken
  // only when the per-element columns are at most an eighth of a row.
  if (m == 2 && !any_b1 && shift_tier && !pl->stores.empty()) {
    bool ok = ms[0] < (int64_t(1) << 30);
    int64_t sp = -1;
    for (size_t i = 0; i < all.size() && ok; ++i)
      if (wst[i][1] != 1 || wst[i][0] % 4 != 0) ok = false;
    for (const View& v : pl->stores) {
      const int64_t ph = (int64_t)((reinterpret_cast<uintptr_t>(v.ptr) / (uintptr_t)elem_size(v.dtype)) % 4);
      if (sp < 0) sp = ph;
      else if (ph != sp) ok = false;
    }
    const int64_t head = (4 - sp) % 4 + 4;
    const int64_t W = cmdx::contig_chunk(P.tier, P.extended, false);
    const int64_t cols = ms[1];
    const int64_t main_cols = cols >= head + 4 ? (cols - head - 4) / W * W : 0;
    if (ok && main_cols > 0 && 8 * (cols - main_cols) <= cols && main_cols / W < (int64_t(1) << 30)) {
      pl->path = CMD_PATH_CONTIG;
      pl->rows = ms[0];
      pl->head = head;
      pl->shifted = true;
      return CMD_OK;
    }
  }
  pl->path = CMD_PATH_GENERIC;
  return CMD_OK;
}

// Magic number of the Granlund-Montgomery round-up division for 64-bit
// dividends: l = ceil(log2 d), m = floor(2^64 (2^l - d) / d) + 1.
cmdx::FastDiv make_fastdiv(int64_t d) {
  cmdx::FastDiv f{};
  f.d = d;
  if (d <= 1) return f;
  uint32_t l = 0;
  while (l < 63 && (int64_t(1) << l) < d) ++l;
  if ((int64_t(1) << l) < d) l = 64;
  unsigned __int128 two_l = (unsigned __int128)1 << l;
  unsigned __int128 m = (((unsigned __int128)1 << 64) * (two_l - (unsigned __int128)d)) / (unsigned __int128)d + 1;
  f.m = (uint64_t)m;
  f.l = l;
  return f;
}

cmd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CMD_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

}  // namespace

namespace cmdx {

void set_last_error(cmd_status s, const char* msg) { fail(s, msg); }

// cmd_compile without the device allocation: the kernel's error word is
// words[slot] of a caller-provided static device array of `capacity` words.
cmd_status compile_with_static_word(cmd_command_t cmd, cmd_kernel_t* out, uint32_t* words, int capacity) {
  if (!cmd || !out) return fail(CMD_ERR_NULL, "cmd or out is NULL");
  cmd_kernel* k = new (std::nothrow) cmd_kernel();
  if (!k) return fail(CMD_ERR_NOMEM, "out of host memory");
  try {
    k->ops = cmd->ops;
    cmd_status s = check_command(cmd, &k->rank);
    if (s == CMD_OK) s = lower(k->ops, &k->prog);
    if (s != CMD_OK) {
      delete k;
      return s;
    }
  } catch (...) {
    delete k;
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    delete k;
    return cuda_fail(e, "cudaGetDevice");
  }
  bool reused = false;
  const int slot = acquire_slot(dev, &reused);
  if (slot < 0) {
    delete k;
    return fail(CMD_ERR_LIMIT, "more than " + std::to_string(CMD_MAX_KERNELS) + " compiled kernels on this device");
  }
  if (slot >= capacity) {
    release_slot(dev, slot);
    delete k;
    return fail(CMD_ERR_LIMIT, "the static scratch array holds " + std::to_string(capacity) +
                                   " error words; program slot " + std::to_string(slot) + " is beyond it");
  }
  if (reused) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cmdx::upload_program(k->prog.tier, k->prog.extended, slot, k->prog.words.data(), (int)k->prog.words.size());
  // the word keeps whatever the previous kernel in this slot left: clear it
  if (e == cudaSuccess) e = clear_device_now(words + slot, sizeof(uint32_t));
  if (e != cudaSuccess) {
    release_slot(dev, slot);
    delete k;
    return cuda_fail(e, "uploading the program / clearing the static error word");
  }
  k->err = words + slot;
  k->err_owned = false;
  k->device = dev;
  k->slot = slot;
  *out = k;
  return CMD_OK;
}

}  // namespace cmdx

// ============================================================================
// C ABI
// ============================================================================

extern "C" {

int32_t cmd_abi_version(void) { return CMD_ABI_VERSION; }

const char* cmd_status_string(cmd_status s) {
  switch (s) {
    case CMD_OK: return "CMD_OK";
    case CMD_ERR_NULL: return "CMD_ERR_NULL";
    case CMD_ERR_BAD_TAG: return "CMD_ERR_BAD_TAG";
    case CMD_ERR_TYPE: return "CMD_ERR_TYPE";
    case CMD_ERR_SHAPE: return "CMD_ERR_SHAPE";
    case CMD_ERR_ALIAS: return "CMD_ERR_ALIAS";
    case CMD_ERR_ALIGN: return "CMD_ERR_ALIGN";
    case CMD_ERR_STATE: return "CMD_ERR_STATE";
    case CMD_ERR_LIMIT: return "CMD_ERR_LIMIT";
    case CMD_ERR_CUDA: return "CMD_ERR_CUDA";
    case CMD_ERR_DEVICE_TIMEOUT: return "CMD_ERR_DEVICE_TIMEOUT";
    case CMD_ERR_NOMEM: return "CMD_ERR_NOMEM";
    case CMD_ERR_ARG: return "CMD_ERR_ARG";
  }
  return "CMD_ERR_UNKNOWN";
}

const char* cmd_last_error(void) { return g_last_error.c_str(); }

cmd_status cmd_create(cmd_command_t* out) {
  if (!out) return fail(CMD_ERR_NULL, "out is NULL");
  cmd_command* c = new (std::nothrow) cmd_command();
  if (!c) return fail(CMD_ERR_NOMEM, "out of host memory");
  *out = c;
  return CMD_OK;
}

void cmd_destroy(cmd_command_t cmd) { delete cmd; }

cmd_status cmd_next_tag(cmd_command_t cmd, cmd_tag* out) {
  if (!cmd || !out) return fail(CMD_ERR_NULL, "cmd or out is NULL");
  *out = (cmd_tag)cmd->ops.size();
  return CMD_OK;
}

static cmd_status push_op(cmd_command_t cmd, const Op& op, cmd_tag* out) {
  if (cmd->ops.size() >= (size_t)CMD_MAX_TAGS)
    return fail(CMD_ERR_LIMIT, "a Command holds at most " + std::to_string(CMD_MAX_TAGS) + " operations");
  try {
    cmd->ops.push_back(op);
  } catch (...) {
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  if (out) *out = (cmd_tag)(cmd->ops.size() - 1);
  return CMD_OK;
}

cmd_status cmd_add_load_tensor(cmd_command_t cmd, cmd_dtype dtype, int32_t rank, cmd_tag* out) {
  if (!cmd) return fail(CMD_ERR_NULL, "cmd is NULL");
  if (!valid_dtype(dtype)) return fail(CMD_ERR_TYPE, "unknown dtype " + std::to_string((int)dtype));
  if (rank < 0 || rank > CMD_MAX_RANK) return fail(CMD_ERR_SHAPE, "rank must be 0.." + std::to_string(CMD_MAX_RANK));
  Op op{kLoad, (int)dtype, rank, 0, -1, -1, -1, dtype == CMD_I32 ? kInt : kFloat};
  return push_op(cmd, op, out);
}

cmd_status cmd_add_load_scalar(cmd_command_t cmd, cmd_dtype dtype, cmd_tag* out) {
  if (!cmd) return fail(CMD_ERR_NULL, "cmd is NULL");
  if (dtype != CMD_F32 && dtype != CMD_I32)
    return fail(CMD_ERR_TYPE, "a Load_Scalar is CMD_F32 or CMD_I32");
  Op op{kScalar, (int)dtype, 0, 0, -1, -1, -1, dtype == CMD_I32 ? kInt : kFloat};
  return push_op(cmd, op, out);
}

cmd_status cmd_add_execute(cmd_command_t cmd, const cmd_xop* ops, int32_t n, cmd_tag* out_tags) {
  if (!cmd || !ops) return fail(CMD_ERR_NULL, "cmd or ops is NULL");
  if (n <= 0) return fail(CMD_ERR_ARG, "a T_Execute block needs at least one E op");
  const int base = (int)cmd->ops.size();
  if (base + n > CMD_MAX_TAGS)
    return fail(CMD_ERR_LIMIT, "a Command holds at most " + std::to_string(CMD_MAX_TAGS) + " operations");
  std::vector<Op> block;
  auto resolve = [&](cmd_tag t, int i, int* res) -> cmd_status {
    if (t < 0) {
      int li = -1 - t;
      if (li >= i)
        return fail(CMD_ERR_BAD_TAG, "E op " + std::to_string(i) + " refers to CMD_LOCAL(" + std::to_string(li) +
                                         "), which is not an earlier op of the block");
      *res = base + li;
      return CMD_OK;
    }
    if (t >= base)
      return fail(CMD_ERR_BAD_TAG, "E op " + std::to_string(i) + " refers to tag " + std::to_string(t) +
                                       ", which does not exist yet (use CMD_LOCAL for results of this block)");
    if (cmd->ops[t].kind == kStore)
      return fail(CMD_ERR_BAD_TAG, "E op " + std::to_string(i) + " refers to tag " + std::to_string(t) +
                                       ", a Store_Tensor, which has no value");
    *res = t;
    return CMD_OK;
  };
  auto cls_of = [&](int t) { return t < base ? cmd->ops[t].cls : block[t - base].cls; };
  for (int i = 0; i < n; ++i) {
    const cmd_xop& x = ops[i];
    if (x.op < CMD_E_ADD || x.op > CMD_E_SELECT) return fail(CMD_ERR_ARG, "unknown E op " + std::to_string(x.op));
    Op op{kExec, 0, 0, x.op, -1, -1, -1, kFloat};
    if (cmd_status s = resolve(x.a, i, &op.a)) return s;
    if (!is_unary(x.op)) {
      if (cmd_status s = resolve(x.b, i, &op.b)) return s;
      if (cls_of(op.a) != cls_of(op.b))
        return fail(CMD_ERR_TYPE, "E op " + std::to_string(i) + " mixes an int value and a float value");
    }
    if (x.op >= CMD_E_ULT && x.op <= CMD_E_UGE && cls_of(op.a) != kInt)
      return fail(CMD_ERR_TYPE, "E op " + std::to_string(i) + ": unsigned comparisons take int values");
    if (x.op == CMD_E_SELECT) {
      if (cmd_status s = resolve(x.c, i, &op.c)) return s;
      if (cls_of(op.c) != kInt)
        return fail(CMD_ERR_TYPE, "E op " + std::to_string(i) + ": the condition of a SELECT must be int-valued");
    }
    op.cls = x.op == CMD_E_TO_F32 ? kFloat : (x.op == CMD_E_TO_I32 || is_compare(x.op)) ? kInt : cls_of(op.a);
    op.block = cmd->n_blocks;
    block.push_back(op);
  }
  try {
    cmd->ops.insert(cmd->ops.end(), block.begin(), block.end());
  } catch (...) {
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  ++cmd->n_blocks;
  if (out_tags)
    for (int i = 0; i < n; ++i) out_tags[i] = base + i;
  return CMD_OK;
}

cmd_status cmd_add_store(cmd_command_t cmd, cmd_tag src, cmd_dtype dtype, int32_t rank, cmd_tag* out) {
  if (!cmd) return fail(CMD_ERR_NULL, "cmd is NULL");
  if (!valid_store_dtype(dtype)) return fail(CMD_ERR_TYPE, "unknown dtype " + std::to_string((int)dtype));
  if (rank < 0 || rank > CMD_MAX_RANK) return fail(CMD_ERR_SHAPE, "rank must be 0.." + std::to_string(CMD_MAX_RANK));
  if (src < 0 || src >= (cmd_tag)cmd->ops.size() || cmd->ops[src].kind == kStore)
    return fail(CMD_ERR_BAD_TAG, "store source tag " + std::to_string(src) + " is not an earlier value");
  const int cls = cmd->ops[src].cls;
  if ((dtype == CMD_I32 || dtype == CMD_B1) != (cls == kInt))
    return fail(CMD_ERR_TYPE, std::string("cannot store a ") + (cls == kInt ? "int" : "float") + " value as " +
                                  dtype_name(dtype));
  Op op{kStore, (int)dtype, rank, 0, src, -1, -1, kNone};
  return push_op(cmd, op, out);
}

cmd_status cmd_lower(cmd_command_t cmd, cmd_program_info* info, uint32_t* words, int32_t cap) {
  if (!cmd || !info) return fail(CMD_ERR_NULL, "cmd or info is NULL");
  int rank;
  if (cmd_status s = check_command(cmd, &rank)) return s;
  Program P;
  try {
    if (cmd_status s = lower(cmd->ops, &P)) return s;
  } catch (...) {
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  fill_info(P, info);
  if (words)
    for (int i = 0; i < cap && i < (int)P.words.size(); ++i) words[i] = P.words[i];
  return CMD_OK;
}

cmd_status cmd_compile(cmd_command_t cmd, cmd_kernel_t* out) {
  if (!cmd || !out) return fail(CMD_ERR_NULL, "cmd or out is NULL");
  cmd_kernel* k = new (std::nothrow) cmd_kernel();
  if (!k) return fail(CMD_ERR_NOMEM, "out of host memory");
  try {
    k->ops = cmd->ops;
    if (cmd_status s = check_command(cmd, &k->rank)) {
      delete k;
      return s;
    }
    if (cmd_status s = lower(k->ops, &k->prog)) {
      delete k;
      return s;
    }
  } catch (...) {
    delete k;
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    delete k;
    return cuda_fail(e, "cudaGetDevice");
  }
  bool reused = false;
  int slot = acquire_slot(dev, &reused);
  if (slot < 0) {
    delete k;
    return fail(CMD_ERR_LIMIT, "more than " + std::to_string(CMD_MAX_KERNELS) + " compiled kernels on this device");
  }
  if (reused) {
    // a destroyed kernel's launches may still read this slot
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      release_slot(dev, slot);
      delete k;
      return cuda_fail(e, "cudaDeviceSynchronize before reusing a program slot");
    }
  }
  e = cmdx::upload_program(k->prog.tier, k->prog.extended, slot, k->prog.words.data(), (int)k->prog.words.size());
  if (e == cudaSuccess) {
    e = cudaMalloc(&k->err, 256);
    if (e == cudaSuccess) g_device_allocs.fetch_add(1);
  }
  if (e == cudaSuccess) e = clear_device_now(k->err, 256);
  if (e != cudaSuccess) {
    if (k->err) cudaFree(k->err);
    release_slot(dev, slot);
    delete k;
    return cuda_fail(e, "uploading the program / allocating the device error word");
  }
  k->device = dev;
  k->slot = slot;
  *out = k;
  return CMD_OK;
}

cmd_status cmd_lower_kernel(cmd_command_t cmd, cmd_kernel_t* out) {
  if (!cmd || !out) return fail(CMD_ERR_NULL, "cmd or out is NULL");
  cmd_kernel* k = new (std::nothrow) cmd_kernel();
  if (!k) return fail(CMD_ERR_NOMEM, "out of host memory");
  try {
    k->ops = cmd->ops;
    cmd_status s = check_command(cmd, &k->rank);
    if (s == CMD_OK) s = lower(k->ops, &k->prog);
    if (s != CMD_OK) {
      delete k;
      return s;
    }
  } catch (...) {
    delete k;
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  *out = k;
  return CMD_OK;
}

void cmd_kernel_destroy(cmd_kernel_t k) {
  if (!k) return;
  if (k->err && k->err_owned) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != k->device) cudaSetDevice(k->device);
    cudaFree(k->err);
    if (cur != k->device && cur >= 0) cudaSetDevice(cur);
  }
  if (k->slot >= 0) release_slot(k->device, k->slot);
  delete k;
}

cmd_status cmd_kernel_info(cmd_kernel_t k, cmd_program_info* info) {
  if (!k || !info) return fail(CMD_ERR_NULL, "k or info is NULL");
  fill_info(k->prog, info);
  return CMD_OK;
}

cmd_status cmd_to_yaml(cmd_command_t cmd, char* buf, int64_t size, int64_t* needed) {
  if (!cmd) return fail(CMD_ERR_NULL, "cmd is NULL");
  std::string s;
  try {
    s += "# tensor Command, text form (YAML)\nversion: 1\noperations:\n";
    char line[200];
    const auto& ops = cmd->ops;
    for (size_t t = 0; t < ops.size(); ++t) {
      const Op& op = ops[t];
      switch (op.kind) {
        case kLoad:
          std::snprintf(line, sizeof line, "  - {kind: load_tensor, tag: %zu, dtype: %s, rank: %d}\n", t,
                        dtype_name(op.dtype), op.rank);
          s += line;
          break;
        case kScalar:
          std::snprintf(line, sizeof line, "  - {kind: load_scalar, tag: %zu, dtype: %s}\n", t, dtype_name(op.dtype));
          s += line;
          break;
        case kStore:
          std::snprintf(line, sizeof line, "  - {kind: store_tensor, tag: %zu, src: %d, dtype: %s, rank: %d}\n", t,
                        op.a, dtype_name(op.dtype), op.rank);
          s += line;
          break;
        default:
          if (t == 0 || ops[t - 1].kind != kExec || ops[t - 1].block != op.block) s += "  - kind: execute\n    ops:\n";
          if (is_unary(op.eop))
            std::snprintf(line, sizeof line, "      - {tag: %zu, op: %s, a: %d}\n", t, eop_name(op.eop), op.a);
          else if (op.eop == CMD_E_SELECT)
            std::snprintf(line, sizeof line, "      - {tag: %zu, op: %s, a: %d, b: %d, c: %d}\n", t,
                          eop_name(op.eop), op.a, op.b, op.c);
          else
            std::snprintf(line, sizeof line, "      - {tag: %zu, op: %s, a: %d, b: %d}\n", t, eop_name(op.eop),
                          op.a, op.b);
          s += line;
          break;
      }
    }
  } catch (...) {
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  if (needed) *needed = (int64_t)s.size() + 1;
  if (buf && size > 0) {
    size_t n = std::min<size_t>((size_t)size - 1, s.size());
    std::memcpy(buf, s.data(), n);
    buf[n] = 0;
  }
  return CMD_OK;
}

cmd_status cmd_kernel_dump(cmd_kernel_t k, char* buf, int64_t size, int64_t* needed) {
  if (!k) return fail(CMD_ERR_NULL, "k is NULL");
  static const char* bin[] = {"fadd", "fsub", "frsub", "fmul", "iadd", "isub", "irsub", "imul",
                              "fdiv", "frdiv", "idiv", "irdiv", "fmin", "fmax", "imin", "imax"};
  static const char* un[] = {"fneg", "ineg", "mov", "fabs", "iabs", "i2f", "f2i"};
  static const char* cmp[] = {"flt", "fle", "fgt", "fge", "feq", "fne", "ilt", "ile",
                              "igt", "ige", "ieq", "ine", "ult", "ule", "ugt", "uge"};
  std::string s;
  const Program& P = k->prog;
  char line[160];
  std::snprintf(line, sizeof line, "; tier %d, %d slots, %d words, %d live E ops, %d moves\n", P.tier, P.n_slots,
                (int)P.words.size(), P.n_live_e, P.n_moves);
  s += line;
  for (size_t j = 0; j < P.load_tags.size(); ++j) {
    std::snprintf(line, sizeof line, "load    r%zu <- tag %d (%s)\n", j, P.load_tags[j],
                  dtype_name(k->ops[P.load_tags[j]].dtype));
    s += line;
  }
  for (size_t j = 0; j < P.scalar_tags.size(); ++j) {
    std::snprintf(line, sizeof line, "scalar  s%zu <- tag %d (%s)\n", j, P.scalar_tags[j],
                  dtype_name(k->ops[P.scalar_tags[j]].dtype));
    s += line;
  }
  for (size_t i = 0; i < P.code.size(); ++i) {
    const Instr& in = P.code[i];
    switch (in.kind) {
      case Instr::kBin: std::snprintf(line, sizeof line, "%-7s r%d, r%d\n", bin[in.op], in.d, in.s); break;
      case Instr::kUn: std::snprintf(line, sizeof line, "%-7s r%d, r%d\n", un[in.op], in.d, in.s); break;
      case Instr::kBinS: std::snprintf(line, sizeof line, "%-7s r%d, s%d\n", bin[in.op], in.d, in.aux); break;
      case Instr::kMovS: std::snprintf(line, sizeof line, "mov     r%d, s%d\n", in.d, in.aux); break;
      case Instr::kSDiv: {
        const int own = P.derived[in.aux - (int)P.scalar_tags.size()].second;
        std::snprintf(line, sizeof line, "%s r%d, s%d  ; through s%d..s%d, derived from s%d at launch\n",
                      in.op == 0 ? "fdivs  " : "idivs  ", in.d, own, in.aux, in.aux + (in.op == 0 ? 1 : 2), own);
        break;
      }
      case Instr::kCmpX:
        std::snprintf(line, sizeof line, "%-7s r%d, r%d\n", cmp[in.op], in.d, cmdx::tier_slots(P.tier) - 1);
        break;
      case Instr::kCmpS: std::snprintf(line, sizeof line, "%-7s r%d, s%d\n", cmp[in.op], in.d, in.aux); break;
      case Instr::kSel:
        std::snprintf(line, sizeof line, "sel     r%d, r%d  ; r%d = r%d != 0 ? r%d : r%d\n", in.d, in.s, in.d,
                      cmdx::tier_slots(P.tier) - 1, in.d, in.s);
        break;
      case Instr::kSelS:
        std::snprintf(line, sizeof line, "sel     r%d, s%d  ; r%d = r%d != 0 ? r%d : s%d\n", in.d, in.aux, in.d,
                      cmdx::tier_slots(P.tier) - 1, in.d, in.aux);
        break;
      case Instr::kSt:
        std::snprintf(line, sizeof line, "store   out%d <- r%d (%s, tag %d)\n", in.aux, in.s, dtype_name(in.op),
                      P.store_tags[in.aux]);
        break;
    }
    s += line;
  }
  s += "end\n";
  if (needed) *needed = (int64_t)s.size() + 1;
  if (buf && size > 0) {
    size_t n = std::min<size_t>((size_t)size - 1, s.size());
    std::memcpy(buf, s.data(), n);
    buf[n] = 0;
  }
  return CMD_OK;
}

// How a contiguous plan splits: the warp chunk of the kernel it runs, the
// columns of a row walk (the elements of a dense range), and the elements
// the contiguous kernel covers from `head` on (of every row for a row walk;
// a shifted launch leaves at least 4 after them).
namespace {
struct ContigSplit {
  bool half2;
  int64_t chunk, cols, n_main;
};

ContigSplit contig_split(const Plan& pl, const Program& P) {
  ContigSplit c;
  c.half2 = !pl.shifted && !pl.loads.empty();
  for (const auto& v : pl.loads) c.half2 = c.half2 && (v.dtype == CMD_F16 || v.dtype == CMD_BF16);
  c.chunk = cmdx::contig_chunk(P.tier, P.extended, c.half2);
  c.cols = pl.rows > 1 ? pl.msizes[cmdx::kMaxRank - 1] : pl.n;
  c.n_main = pl.shifted ? (c.cols - pl.head - 4) / c.chunk * c.chunk
                        : (c.cols - pl.head) - (c.cols - pl.head) % c.chunk;
  return c;
}

// Elements load j's first contiguous element sits past a vector boundary
// (0 unless the launch is shifted).
int load_shift(const Plan& pl, size_t j) {
  if (!pl.shifted) return 0;
  const int64_t es = elem_size(pl.loads[j].dtype);
  return (int)(((reinterpret_cast<uintptr_t>(pl.loads[j].ptr) / (uintptr_t)es) + (uintptr_t)pl.head) % 4);
}
}  // namespace

cmd_status cmd_plan_launch(cmd_kernel_t k, const cmd_runtime_args* args, cmd_launch_plan* plan) {
  if (!k || !plan) return fail(CMD_ERR_NULL, "k or plan is NULL");
  Plan pl;
  try {
    if (cmd_status s = plan_launch(k, args, &pl)) return s;
  } catch (...) {
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  plan->path = pl.path;
  plan->merged_rank = pl.mrank;
  for (int d = 0; d < CMD_MAX_RANK; ++d) plan->merged_sizes[d] = 1;
  for (int q = 0; q < pl.mrank; ++q) plan->merged_sizes[q] = pl.msizes[cmdx::kMaxRank - pl.mrank + q];
  plan->n_elements = pl.n;
  plan->bytes = pl.bytes;
  plan->n_transposed = pl.n_trans;
  plan->head_elements = 0;
  plan->contig_elements = 0;
  plan->shifted_loads = 0;
  if (pl.path == CMD_PATH_CONTIG) {
    const ContigSplit c = contig_split(pl, k->prog);
    plan->head_elements = pl.head;
    plan->contig_elements = c.n_main;
    for (size_t j = 0; j < pl.loads.size(); ++j) plan->shifted_loads += load_shift(pl, j) != 0;
  }
  return CMD_OK;
}

cmd_status cmd_launch(cmd_kernel_t k, const cmd_runtime_args* args, void* cuda_stream) {
  if (!k) return fail(CMD_ERR_NULL, "k is NULL");
  if (k->slot < 0) return fail(CMD_ERR_STATE, "kernel was lowered without a device (cmd_lower_kernel); compile it");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != k->device)
    return fail(CMD_ERR_STATE, "kernel was compiled for device " + std::to_string(k->device) +
                                   " but device " + std::to_string(dev) + " is current");
  Plan pl;
  try {
    if (cmd_status s = plan_launch(k, args, &pl)) return s;
  } catch (...) {
    return fail(CMD_ERR_NOMEM, "out of host memory");
  }
  if (pl.path == CMD_PATH_NONE) return CMD_OK;
  // A load anywhere but in device memory (pinned or other host memory,
  // managed memory) never takes the tile executor, whose loads are TMA
  // copies that this library issues on device memory only; the generic
  // executor reads the same views with plain loads.
  if (pl.path == CMD_PATH_TILE2D) {
    for (const View& v : pl.loads) {
      cudaPointerAttributes a;
      if (cudaPointerGetAttributes(&a, v.ptr) != cudaSuccess) {
        cudaGetLastError();  // (an unknown pointer: left to the launch)
        continue;
      }
      if (a.type != cudaMemoryTypeDevice) {
        pl.path = CMD_PATH_GENERIC;
        break;
      }
    }
  }
  const Program& P = k->prog;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (pl.path == CMD_PATH_CONTIG) {
    // whole warp chunks on the contiguous executor; a head (the elements
    // before every pointer is vector-aligned) and a ragged tail (fewer than
    // one chunk of elements) on the generic one
    const ContigSplit split = contig_split(pl, P);
    const bool half2 = split.half2;
    const int64_t chunk = split.chunk, cols = split.cols, n_main = split.n_main;
    const int64_t head = pl.head;
    // the generic executor over the 1-D elements [start, start + count),
    // skipping [start + gap_at, start + gap_at + gap)
    auto generic_range = [&](int64_t start, int64_t count, int64_t gap_at, int64_t gap) -> cudaError_t {
      cmdx::GenericParams p;
      std::memset(&p, 0, sizeof p);
      for (size_t j = 0; j < pl.loads.size(); ++j) {
        p.in[j] = static_cast<const char*>(pl.loads[j].ptr) + start * elem_size(pl.loads[j].dtype);
        p.in_dt[j] = (uint8_t)pl.loads[j].dtype;
        p.in_st[j][cmdx::kMaxRank - 1] = 1;
      }
      for (size_t j = 0; j < pl.stores.size(); ++j) {
        // (packed bits have no head, and the tail starts at a multiple of
        // the chunk, so on a word)
        const int64_t skip = pl.stores[j].dtype == CMD_B1 ? start / 8 : start * elem_size(pl.stores[j].dtype);
        p.out[j] = static_cast<char*>(pl.stores[j].ptr) + skip;
        p.out_st[j][cmdx::kMaxRank - 1] = 1;
      }
      for (int d = 0; d < cmdx::kMaxRank; ++d) p.div[d] = make_fastdiv(1);
      p.div[cmdx::kMaxRank - 1] = make_fastdiv(count);
      p.top = cmdx::kMaxRank - 1;
      p.gap_at = gap_at;
      p.gap = gap;
      std::memcpy(p.scal, pl.scal, sizeof p.scal);
      p.n = count;
      p.prog = (uint32_t)k->slot;
      p.n_loads = (uint32_t)pl.loads.size();
      return cmdx::generic_launch(P.tier, P.extended, p, stream);
    };
    e = cudaSuccess;
    if (e == cudaSuccess && n_main > 0) {
      cmdx::ContigParams p;
      std::memset(&p, 0, sizeof p);
      for (size_t j = 0; j < pl.loads.size(); ++j) {
        const int64_t es = elem_size(pl.loads[j].dtype);
        p.in[j] = static_cast<const char*>(pl.loads[j].ptr) + head * es;
        p.in_dt[j] = (uint8_t)pl.loads[j].dtype;
        if (pl.shifted) {
          p.in_shift[j] = (uint8_t)load_shift(pl, j);
          p.shifted = 1;
        }
      }
      for (size_t j = 0; j < pl.stores.size(); ++j)
        p.out[j] = static_cast<char*>(pl.stores[j].ptr) + head * elem_size(pl.stores[j].dtype);
      std::memcpy(p.scal, pl.scal, sizeof p.scal);
      p.n = pl.rows > 1 ? pl.rows * n_main : n_main;
      p.prog = (uint32_t)k->slot;
      p.n_loads = (uint32_t)pl.loads.size();
      if (pl.rows > 1) {
        // merged dims are right-aligned: the row dim is the second to last
        const int rd = cmdx::kMaxRank - 2;
        p.rows = (int32_t)pl.rows;
        p.row_chunks = (int32_t)(n_main / chunk);
        for (size_t j = 0; j < pl.loads.size(); ++j) p.in_ld[j] = pl.ml[j][rd];
        for (size_t j = 0; j < pl.stores.size(); ++j) p.out_ld[j] = pl.ms[j][rd];
      }
      bool bits_only = !pl.stores.empty();
      for (const auto& v : pl.stores) bits_only = bits_only && v.dtype == CMD_B1;
      e = cmdx::contig_launch(P.tier, P.extended, p, stream, bits_only, half2);
    }
    // the tail from where the contiguous launch ends; with a head, head and
    // tail in one launch whose index space skips the contiguous launch's
    // elements (there are no packed-bit stores then: those index words by
    // the launch's own element index). A row walk with shifted loads leaves
    // each row's first `head` and last columns: two launches over those
    // column ranges of every row.
    if (pl.rows > 1 && pl.shifted) {
      auto generic_cols = [&](int64_t c0, int64_t nc) -> cudaError_t {
        cmdx::GenericParams p;
        std::memset(&p, 0, sizeof p);
        const int rd = cmdx::kMaxRank - 2;
        for (size_t j = 0; j < pl.loads.size(); ++j) {
          p.in[j] = static_cast<const char*>(pl.loads[j].ptr) + c0 * elem_size(pl.loads[j].dtype);
          p.in_dt[j] = (uint8_t)pl.loads[j].dtype;
          p.in_st[j][rd] = pl.ml[j][rd];
          p.in_st[j][rd + 1] = 1;
        }
        for (size_t j = 0; j < pl.stores.size(); ++j) {
          p.out[j] = static_cast<char*>(pl.stores[j].ptr) + c0 * elem_size(pl.stores[j].dtype);
          p.out_st[j][rd] = pl.ms[j][rd];
          p.out_st[j][rd + 1] = 1;
        }
        for (int d = 0; d < cmdx::kMaxRank; ++d) p.div[d] = make_fastdiv(1);
        p.div[rd] = make_fastdiv(pl.rows);
        p.div[rd + 1] = make_fastdiv(nc);
        p.n = pl.rows * nc;
        p.gap_at = p.n;  // no gap
        p.top = (uint32_t)rd;
        std::memcpy(p.scal, pl.scal, sizeof p.scal);
        p.prog = (uint32_t)k->slot;
        p.n_loads = (uint32_t)pl.loads.size();
        return cmdx::generic_launch(P.tier, P.extended, p, stream);
      };
      if (e == cudaSuccess) e = generic_cols(0, head);
      if (e == cudaSuccess) e = generic_cols(head + n_main, cols - head - n_main);
    } else if (e == cudaSuccess && pl.n > n_main && pl.rows <= 1) {
      e = head == 0 ? generic_range(n_main, pl.n - n_main, pl.n, 0) : generic_range(0, pl.n - n_main, head, n_main);
    }
  } else if (pl.path == CMD_PATH_TILE2D) {
    cmdx::Tile2dLaunch L;
    std::memset(&L, 0, sizeof L);
    const int off = cmdx::kMaxRank - pl.mrank;  // merged dims are right-aligned in ml/ms
    const int row = off + pl.tile_row, col = off + pl.tile_col;
    // batch dims b0 (outer), b1: a single batch dim is b1
    const int b0 = pl.n_batch == 2 ? off + pl.batch[0] : -1;
    const int b1 = pl.n_batch >= 1 ? off + pl.batch[pl.n_batch - 1] : -1;
    for (size_t j = 0; j < pl.loads.size(); ++j) {
      L.in[j] = pl.loads[j].ptr;
      L.in_dt[j] = (uint8_t)pl.loads[j].dtype;
      const bool trans = pl.ml[j][col] != 1;
      L.in_trans[j] = trans;
      L.in_ld[j] = trans ? pl.ml[j][col] : pl.ml[j][row];
      L.in_bst[j][0] = b0 >= 0 ? pl.ml[j][b0] : 0;
      L.in_bst[j][1] = b1 >= 0 ? pl.ml[j][b1] : 0;
    }
    for (size_t j = 0; j < pl.stores.size(); ++j) {
      L.out[j] = pl.stores[j].ptr;
      L.out_ld[j] = pl.ms[j][row];
      L.out_bst[j][0] = b0 >= 0 ? pl.ms[j][b0] : 0;
      L.out_bst[j][1] = b1 >= 0 ? pl.ms[j][b1] : 0;
    }
    std::memcpy(L.scal, pl.scal, sizeof L.scal);
    L.rows = pl.msizes[row];
    L.cols = pl.msizes[col];
    L.nb[0] = b0 >= 0 ? pl.msizes[b0] : 1;
    L.nb[1] = b1 >= 0 ? pl.msizes[b1] : 1;
    L.prog = (uint32_t)k->slot;
    L.n_loads = (uint32_t)pl.loads.size();
    L.err = k->err;
    L.debug = (uint32_t)g_force_timeout.load();
    L.timeout_ns = g_wait_limit_ns.load();
    e = cmdx::tile2d_launch(P.tier, P.extended, L, stream);
  } else {
    cmdx::GenericParams p;
    std::memset(&p, 0, sizeof p);
    for (size_t j = 0; j < pl.loads.size(); ++j) {
      p.in[j] = pl.loads[j].ptr;
      p.in_dt[j] = (uint8_t)pl.loads[j].dtype;
      for (int d = 0; d < cmdx::kMaxRank; ++d) p.in_st[j][d] = pl.ml[j][d];
    }
    for (size_t j = 0; j < pl.stores.size(); ++j) {
      p.out[j] = pl.stores[j].ptr;
      for (int d = 0; d < cmdx::kMaxRank; ++d) p.out_st[j][d] = pl.ms[j][d];
    }
    for (int d = 0; d < cmdx::kMaxRank; ++d) p.div[d] = make_fastdiv(pl.msizes[d]);
    p.gap_at = pl.n;  // no gap
    p.top = cmdx::kMaxRank - 1;
    for (int d = cmdx::kMaxRank - 1; d >= 0; --d)
      if (pl.msizes[d] > 1) p.top = (uint32_t)d;
    std::memcpy(p.scal, pl.scal, sizeof p.scal);
    p.n = pl.n;
    p.prog = (uint32_t)k->slot;
    p.n_loads = (uint32_t)pl.loads.size();
    e = cmdx::generic_launch(P.tier, P.extended, p, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return CMD_OK;
}

cmd_status cmd_sync_status(cmd_kernel_t k, void* cuda_stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "work on the stream failed");
  if (k && k->err) {
    uint32_t word = 0;
    e = cudaMemcpy(&word, k->err, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word) {
      // cleared on the caller's stream, and waited for, so that a launch
      // queued there next finds it clear
      cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
      e = cudaMemsetAsync(k->err, 0, sizeof word, st);
      if (e == cudaSuccess) e = cudaStreamSynchronize(st);
      if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
      std::string what;
      if (word & 1u) what += " consumer-wait";
      if (word & 2u) what += " producer-wait";
      if (word & 4u) what += " drain-wait";
      if (word & 8u) what += " forced-wait";
      return fail(CMD_ERR_DEVICE_TIMEOUT, "a device-side wait gave up after its time limit:" + what +
                                              " (error word 0x" + [&] {
                                                char b[16];
                                                std::snprintf(b, sizeof b, "%x", word);
                                                return std::string(b);
                                              }() + ")");
    }
  }
  return CMD_OK;
}

int64_t cmd_device_allocations(void) { return g_device_allocs.load(); }

cmd_status cmd_configure_waits(uint64_t timeout_ns, int32_t force_timeout) {
  if (timeout_ns == 0) return fail(CMD_ERR_ARG, "timeout_ns must be > 0");
  g_wait_limit_ns.store(timeout_ns);
  g_force_timeout.store(force_timeout ? 1 : 0);
  return CMD_OK;
}

}  // extern "C"
