// cmd_yaml.cpp - cmd_from_yaml: a Command from its text form.
//
// rocRoller, "Design Overview", section "Serialization": a Command converts
// to and from YAML. The text form is the fixed subset documented in cmd.h
// (written by cmd_to_yaml in cmd_api.cpp); this reader accepts exactly that
// subset and rebuilds the Command through the public builder calls, so every
// check of cmd_add_* applies and the rebuilt Command lowers to the same
// program.
#include <cstdint>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "cmd.h"

namespace cmdx {
cmd_status host_fail(cmd_status s, const std::string& msg);
}

namespace {

struct Line {
  int no;       // 1-based line number
  int indent;   // leading spaces
  std::string text;
};

std::string trim(const std::string& s) {
  size_t a = 0, b = s.size();
  while (a < b && (s[a] == ' ' || s[a] == '\t')) ++a;
  while (b > a && (s[b - 1] == ' ' || s[b - 1] == '\t')) --b;
  return s.substr(a, b - a);
}

bool is_token_char(char c) {
  return (c >= 'a' && c <= 'z') || (c >= 'A' && c <= 'Z') || (c >= '0' && c <= '9') || c == '_' || c == '-';
}

bool parse_int(const std::string& v, int32_t* out) {
  if (v.empty() || v.size() > 12) return false;
  size_t i = 0;
  bool neg = false;
  if (v[0] == '-') {
    neg = true;
    i = 1;
  }
  if (i >= v.size()) return false;
  int64_t x = 0;
  for (; i < v.size(); ++i) {
    if (v[i] < '0' || v[i] > '9') return false;
    x = x * 10 + (v[i] - '0');
  }
  if (neg) x = -x;
  if (x < INT32_MIN || x > INT32_MAX) return false;
  *out = (int32_t)x;
  return true;
}

class Reader {
 public:
  explicit Reader(std::vector<Line> lines) : lines_(std::move(lines)) {}

  cmd_status run(cmd_command_t* out) {
    cmd_command_t c = nullptr;
    if (cmd_status s = cmd_create(&c)) return s;
    cmd_status s = build(c);
    if (s != CMD_OK) {
      cmd_destroy(c);
      return s;
    }
    *out = c;
    return CMD_OK;
  }

 private:
  std::vector<Line> lines_;
  size_t pos_ = 0;

  cmd_status err(int line, const std::string& msg) {
    return cmdx::host_fail(CMD_ERR_ARG, "text form, line " + std::to_string(line) + ": " + msg);
  }
  // a builder call failed: keep its status, name the line
  cmd_status builder_err(int line, cmd_status s) {
    return cmdx::host_fail(s, "text form, line " + std::to_string(line) + ": " + cmd_last_error());
  }

  // "{k: v, k: v}" into *m (bare tokens only).
  cmd_status flow_map(const Line& ln, const std::string& t, std::map<std::string, std::string>* m) {
    if (t.size() < 2 || t.front() != '{' || t.back() != '}') return err(ln.no, "expected a {key: value, ...} mapping");
    const std::string body = t.substr(1, t.size() - 2);
    size_t i = 0;
    while (true) {
      while (i < body.size() && body[i] == ' ') ++i;
      if (i >= body.size()) break;
      size_t k0 = i;
      while (i < body.size() && is_token_char(body[i])) ++i;
      std::string key = body.substr(k0, i - k0);
      while (i < body.size() && body[i] == ' ') ++i;
      if (key.empty() || i >= body.size() || body[i] != ':') return err(ln.no, "expected key: value");
      ++i;
      while (i < body.size() && body[i] == ' ') ++i;
      size_t v0 = i;
      while (i < body.size() && is_token_char(body[i])) ++i;
      std::string val = body.substr(v0, i - v0);
      if (val.empty()) return err(ln.no, "missing value for key '" + key + "'");
      if (m->count(key)) return err(ln.no, "key '" + key + "' given twice");
      (*m)[key] = val;
      while (i < body.size() && body[i] == ' ') ++i;
      if (i < body.size()) {
        if (body[i] != ',') return err(ln.no, "expected ',' or '}' after '" + key + ": " + val + "'");
        ++i;
      }
    }
    return CMD_OK;
  }

  cmd_status get_int(const Line& ln, const std::map<std::string, std::string>& m, const char* key, int32_t* v) {
    auto it = m.find(key);
    if (it == m.end()) return err(ln.no, std::string("missing key '") + key + "'");
    if (!parse_int(it->second, v)) return err(ln.no, std::string("'") + key + "' is not an int32: " + it->second);
    return CMD_OK;
  }

  cmd_status get_dtype(const Line& ln, const std::map<std::string, std::string>& m, cmd_dtype* dt) {
    static const std::map<std::string, cmd_dtype> names = {
        {"f32", CMD_F32}, {"f16", CMD_F16}, {"bf16", CMD_BF16}, {"i32", CMD_I32}, {"b1", CMD_B1}};
    auto it = m.find("dtype");
    if (it == m.end()) return err(ln.no, "missing key 'dtype'");
    auto d = names.find(it->second);
    if (d == names.end()) return err(ln.no, "unknown dtype '" + it->second + "'");
    *dt = d->second;
    return CMD_OK;
  }

  cmd_status only_keys(const Line& ln, const std::map<std::string, std::string>& m,
                       std::initializer_list<const char*> keys) {
    for (auto& kv : m) {
      bool ok = false;
      for (const char* k : keys) ok = ok || kv.first == k;
      if (!ok) return err(ln.no, "unexpected key '" + kv.first + "'");
    }
    return CMD_OK;
  }

  cmd_status check_tag(const Line& ln, cmd_command_t c, int32_t tag) {
    cmd_tag next = 0;
    cmd_next_tag(c, &next);
    if (tag != next)
      return err(ln.no, "tag " + std::to_string(tag) + " out of order (the next operation gets tag " +
                            std::to_string(next) + ")");
    return CMD_OK;
  }

  cmd_status build(cmd_command_t c) {
    bool have_version = false, in_ops = false;
    int item_indent = -1;
    while (pos_ < lines_.size()) {
      const Line& ln = lines_[pos_];
      if (!in_ops) {
        if (ln.indent != 0) return err(ln.no, "expected 'version: 1' or 'operations:' at the start of a line");
        if (ln.text.rfind("version:", 0) == 0) {
          int32_t v;
          if (!parse_int(trim(ln.text.substr(8)), &v) || v != 1)
            return err(ln.no, "unsupported version (this reader knows version 1)");
          have_version = true;
        } else if (ln.text == "operations:") {
          if (!have_version) return err(ln.no, "'version: 1' must come before 'operations:'");
          in_ops = true;
        } else {
          return err(ln.no, "unexpected '" + ln.text + "'");
        }
        ++pos_;
        continue;
      }
      // an item of the operations list
      if (ln.text.rfind("- ", 0) != 0) return err(ln.no, "expected a list item '- ...'");
      if (item_indent < 0) item_indent = ln.indent;
      if (ln.indent != item_indent) return err(ln.no, "list items of 'operations' must line up");
      const std::string item = trim(ln.text.substr(2));
      if (item == "kind: execute") {
        if (cmd_status s = execute_block(c, ln)) return s;
        continue;
      }
      std::map<std::string, std::string> m;
      if (cmd_status s = flow_map(ln, item, &m)) return s;
      auto kind = m.find("kind");
      if (kind == m.end()) return err(ln.no, "missing key 'kind'");
      int32_t tag;
      if (cmd_status s = get_int(ln, m, "tag", &tag)) return s;
      if (cmd_status s = check_tag(ln, c, tag)) return s;
      cmd_dtype dt;
      if (kind->second == "load_tensor") {
        int32_t rank;
        if (cmd_status s = only_keys(ln, m, {"kind", "tag", "dtype", "rank"})) return s;
        if (cmd_status s = get_dtype(ln, m, &dt)) return s;
        if (cmd_status s = get_int(ln, m, "rank", &rank)) return s;
        if (cmd_status s = cmd_add_load_tensor(c, dt, rank, nullptr)) return builder_err(ln.no, s);
      } else if (kind->second == "load_scalar") {
        if (cmd_status s = only_keys(ln, m, {"kind", "tag", "dtype"})) return s;
        if (cmd_status s = get_dtype(ln, m, &dt)) return s;
        if (cmd_status s = cmd_add_load_scalar(c, dt, nullptr)) return builder_err(ln.no, s);
      } else if (kind->second == "store_tensor") {
        int32_t src, rank;
        if (cmd_status s = only_keys(ln, m, {"kind", "tag", "src", "dtype", "rank"})) return s;
        if (cmd_status s = get_int(ln, m, "src", &src)) return s;
        if (cmd_status s = get_dtype(ln, m, &dt)) return s;
        if (cmd_status s = get_int(ln, m, "rank", &rank)) return s;
        if (cmd_status s = cmd_add_store(c, src, dt, rank, nullptr)) return builder_err(ln.no, s);
      } else {
        return err(ln.no, "unknown kind '" + kind->second + "'");
      }
      ++pos_;
    }
    if (!have_version) return err(lines_.empty() ? 1 : lines_.back().no, "missing 'version: 1'");
    if (!in_ops) return err(lines_.empty() ? 1 : lines_.back().no, "missing 'operations:'");
    return CMD_OK;
  }

  // "- kind: execute" at lines_[pos_], then "ops:" and its "- {...}" entries.
  cmd_status execute_block(cmd_command_t c, const Line& head) {
    static const std::map<std::string, int> eops = {
        {"add", CMD_E_ADD}, {"sub", CMD_E_SUB}, {"mul", CMD_E_MUL}, {"neg", CMD_E_NEG}, {"div", CMD_E_DIV},
        {"min", CMD_E_MIN}, {"max", CMD_E_MAX}, {"abs", CMD_E_ABS}, {"to_f32", CMD_E_TO_F32},
        {"to_i32", CMD_E_TO_I32}, {"lt", CMD_E_LT}, {"le", CMD_E_LE}, {"gt", CMD_E_GT}, {"ge", CMD_E_GE},
        {"eq", CMD_E_EQ}, {"ne", CMD_E_NE}, {"ult", CMD_E_ULT}, {"ule", CMD_E_ULE}, {"ugt", CMD_E_UGT},
        {"uge", CMD_E_UGE}, {"select", CMD_E_SELECT}};
    const int item_indent = head.indent;
    ++pos_;
    if (pos_ >= lines_.size() || lines_[pos_].indent <= item_indent || lines_[pos_].text != "ops:")
      return err(head.no, "an execute item needs an indented 'ops:' line after it");
    const int ops_indent = lines_[pos_].indent;
    ++pos_;
    cmd_tag base = 0;
    cmd_next_tag(c, &base);
    std::vector<cmd_xop> xs;
    int entry_indent = -1;
    while (pos_ < lines_.size() && lines_[pos_].indent > ops_indent) {
      const Line& ln = lines_[pos_];
      if (ln.text.rfind("- ", 0) != 0) return err(ln.no, "expected an E op '- {...}'");
      if (entry_indent < 0) entry_indent = ln.indent;
      if (ln.indent != entry_indent) return err(ln.no, "E ops of one block must line up");
      std::map<std::string, std::string> m;
      if (cmd_status s = flow_map(ln, trim(ln.text.substr(2)), &m)) return s;
      if (cmd_status s = only_keys(ln, m, {"tag", "op", "a", "b", "c"})) return s;
      int32_t tag;
      if (cmd_status s = get_int(ln, m, "tag", &tag)) return s;
      const int32_t want = base + (int32_t)xs.size();
      if (tag != want)
        return err(ln.no, "tag " + std::to_string(tag) + " out of order (this E op gets tag " +
                              std::to_string(want) + ")");
      auto op = m.find("op");
      if (op == m.end()) return err(ln.no, "missing key 'op'");
      auto e = eops.find(op->second);
      if (e == eops.end()) return err(ln.no, "unknown E op '" + op->second + "'");
      cmd_xop x{e->second, -1, -1, -1};
      const bool unary = e->second == CMD_E_NEG || e->second == CMD_E_ABS || e->second == CMD_E_TO_F32 ||
                         e->second == CMD_E_TO_I32;
      // operands: earlier tags; results of this block become CMD_LOCAL refs
      auto operand = [&](const char* key, cmd_tag* dst) -> cmd_status {
        int32_t v;
        if (cmd_status s = get_int(ln, m, key, &v)) return s;
        if (v < 0 || v >= tag)
          return err(ln.no, std::string("operand ") + key + " = " + std::to_string(v) +
                                " does not name an earlier operation");
        *dst = v >= base ? CMD_LOCAL(v - base) : v;
        return CMD_OK;
      };
      if (cmd_status s = operand("a", &x.a)) return s;
      if (unary) {
        if (m.count("b") || m.count("c")) return err(ln.no, "'" + op->second + "' takes one operand, a");
      } else {
        if (cmd_status s = operand("b", &x.b)) return s;
        if (e->second == CMD_E_SELECT) {
          if (cmd_status s = operand("c", &x.c)) return s;
        } else if (m.count("c")) {
          return err(ln.no, "only select takes an operand c");
        }
      }
      xs.push_back(x);
      ++pos_;
    }
    if (xs.empty()) return err(head.no, "an execute item needs at least one E op");
    if (cmd_status s = cmd_add_execute(c, xs.data(), (int32_t)xs.size(), nullptr)) return builder_err(head.no, s);
    return CMD_OK;
  }
};

}  // namespace

extern "C" cmd_status cmd_from_yaml(const char* text, int64_t len, cmd_command_t* out) {
  if (!text || !out) return cmdx::host_fail(CMD_ERR_NULL, "text or out is NULL");
  try {
    const size_t n = len < 0 ? std::strlen(text) : (size_t)len;
    std::vector<Line> lines;
    size_t i = 0;
    int no = 0;
    while (i < n) {
      size_t j = i;
      while (j < n && text[j] != '\n') ++j;
      std::string raw(text + i, j - i);
      ++no;
      i = j + 1;
      if (!raw.empty() && raw.back() == '\r') raw.pop_back();
      // a comment runs from a '#' at the line's start or after a space to the end
      for (size_t k = 0; k < raw.size(); ++k)
        if (raw[k] == '#' && (k == 0 || raw[k - 1] == ' ')) {
          raw.resize(k);
          break;
        }
      if (raw.find('\t') != std::string::npos)
        return cmdx::host_fail(CMD_ERR_ARG, "text form, line " + std::to_string(no) + ": tabs are not allowed");
      const std::string t = trim(raw);
      if (t.empty()) continue;
      size_t ind = 0;
      while (ind < raw.size() && raw[ind] == ' ') ++ind;
      lines.push_back({no, (int)ind, t});
    }
    return Reader(std::move(lines)).run(out);
  } catch (...) {
    return cmdx::host_fail(CMD_ERR_NOMEM, "out of host memory");
  }
}
