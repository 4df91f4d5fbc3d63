/*
 * ks_oracle.cpp — CPU oracle for the warp-level SIMT PTX interpreter.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, by smoke() and by the
 * bench's CPU-baseline / reference legs, never by the product path. It shares
 * no code with the GPU path. It is written to be read against the pages, not
 * to be fast: one C++ struct per simulated lane, instructions kept as parsed
 * records, post-dominators as plain sets, warps interpreted one after another.
 *
 * What it follows (page, then section):
 *  - KernelScope backend doc, simulator/models.py — Thread, Warp, Block: a warp
 *    is 32 threads with a 32-bit active mask and a SIMT stack whose entries are
 *    (pc, active_mask, reconvergence_point); a thread is inactive when its id is
 *    beyond the block size, when it diverged away, or when it exited ("Concepts",
 *    active-mask causes).
 *  - KernelScope backend doc, simulator/engine.py — PtxSimulator.load_kernel /
 *    step / run: blocks of warps, one instruction per warp per step, until every
 *    warp has finished (bounded by a step cap).
 *  - KernelScope backend doc, simulator/engine.py — analyze_global_memory_access:
 *    128-byte lines and 32-byte sectors over the active lanes' addresses.
 *  - KernelScope backend doc, latency/model.py — InstructionTiming: a fixed
 *    latency per instruction class (values supplied by the caller).
 *  - CuTeDSL IKET 浅析 §2 — per-warp slot of a 16-byte header plus
 *    maxTsCntPerWarp records, no cross-warp atomics, overflow counted not lost.
 *  - KernelScope backend doc, simulator/models.py Block (a 48 KB zeroed shared
 *    array and a barrier per block), simulator/engine.py step (warps waiting
 *    at a barrier are skipped) and analyze_shared_memory_access (bank =
 *    (address / 4) % 32; a bank whose lanes all use one address is a
 *    broadcast; otherwise its conflict degree is its number of lanes; the
 *    request's degree, its transactions, is the largest over banks, at least 1).
 *
 * Readings where the pages are silent (each applied identically on the GPU):
 *  - %tid.x is the thread's index in its CTA (the page's `tid % 32` is the lane).
 *  - A divergent branch at pc with immediate post-dominator R: if the top entry
 *    already reconverges at R it is replaced, otherwise its pc becomes R; then
 *    the taken lanes are pushed (unless the target is R) and the fall-through
 *    lanes are pushed last (unless pc+1 is R), so fall-through runs first. An
 *    entry is popped when its pc reaches its reconvergence pc or its mask is
 *    empty. `ret` removes its lanes from every entry.
 *  - Cycles: in-order scoreboard. t = max(t_next, ready[sources], ready[guard],
 *    ready[destinations]); destinations become ready at t + latency; bra and
 *    ret set t_next = t + latency, every other instruction t_next = t + 1; a
 *    store completes at t + latency. cycles = max(last issue + 1, max ready,
 *    last store completion). Trace pseudo-ops cost nothing.
 *  - Sectors: distinct addr>>5 over the executing lanes; lines: distinct addr>>7.
 *  - f32 arithmetic is IEEE binary32 round-to-nearest-even with subnormals;
 *    every NaN result of add/sub/mul/fma/div/sqrt is written as 0x7FFFFFFF.
 *  - Barriers are per warp, as the page's Warp.at_barrier: a warp that issues
 *    bar.sync 0 (any active mask) stops; when every warp of the CTA has
 *    stopped at a barrier or finished, the stopped warps resume with
 *    t_next = (latest bar.sync issue cycle among them) + the bar.sync latency.
 *    A finished warp never holds a barrier. Only barrier 0 without a thread
 *    count, unguarded.
 *  - Shared memory: .shared arrays declared in the kernel body, laid out in
 *    declaration order at their alignment from address 0, at most 48 KiB; a
 *    shared address is a register (32- or 64-bit, zero-extended) or a symbol,
 *    plus an offset. Misaligned (checked first) or out-of-range accesses give
 *    the same statuses as global ones. The bank rule reads each lane's
 *    address only, for 4- and 8-byte accesses alike. ld.shared results are
 *    ready at t + the ld.shared latency; a shared store completes at t + the
 *    st.shared latency. Bank conflicts do not change the timing.
 */
#include "ks_oracle.h"

#include <algorithm>
#include <cctype>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <set>
#include <stdexcept>
#include <string>
#include <thread>
#include <vector>

namespace {

struct OracleError {
  int code;
  std::string msg;
};

[[noreturn]] void fail(int code, int line, const std::string& msg) {
  char buf[64];
  std::snprintf(buf, sizeof buf, "line %d: ", line);
  throw OracleError{code, std::string(buf) + msg};
}

// ---------------------------------------------------------------- types ----

enum Ty { TY_NONE, TY_U32, TY_S32, TY_B32, TY_F32, TY_U64, TY_S64, TY_B64, TY_PRED };

Ty type_from(const std::string& s) {
  if (s == "u32") return TY_U32;
  if (s == "s32") return TY_S32;
  if (s == "b32") return TY_B32;
  if (s == "f32") return TY_F32;
  if (s == "u64") return TY_U64;
  if (s == "s64") return TY_S64;
  if (s == "b64") return TY_B64;
  if (s == "pred") return TY_PRED;
  return TY_NONE;
}

int width_of(Ty t) {
  switch (t) {
    case TY_U32: case TY_S32: case TY_B32: case TY_F32: return 32;
    case TY_U64: case TY_S64: case TY_B64: return 64;
    case TY_PRED: return 1;
    default: return 0;
  }
}

bool is_signed_ty(Ty t) { return t == TY_S32 || t == TY_S64; }
bool is_int_ty(Ty t) { return t == TY_U32 || t == TY_S32 || t == TY_U64 || t == TY_S64; }

// ---------------------------------------------------------- program form ----

enum Kind {
  K_ADD, K_SUB, K_MUL, K_MAD, K_FMA, K_DIV, K_SQRT, K_AND, K_OR, K_XOR, K_SHL, K_SHR,
  K_CVT, K_MOV, K_SETP, K_SELP, K_BRA, K_LDG, K_STG, K_LDP, K_RET, K_EVENT,
  K_LDS, K_STS, K_BAR
};

enum Special { SP_TID_X, SP_TID_Y, SP_TID_Z, SP_NTID_X, SP_NTID_Y, SP_NTID_Z, SP_CTAID_X,
               SP_CTAID_Y, SP_CTAID_Z, SP_NCTAID_X, SP_NCTAID_Y, SP_NCTAID_Z, SP_LANEID };

enum Cmp { C_EQ, C_NE, C_LT, C_LE, C_GT, C_GE };
enum Rnd { R_NONE, R_RN, R_RNI, R_RZI, R_RMI, R_RPI };

struct Opnd {
  enum { NONE, REG, IMM, SPEC, MEM, PARAM, LABEL } k = NONE;
  int reg = -1;        // REG, MEM (base register)
  uint64_t imm = 0;    // IMM bits (already truncated to the operand width)
  int spec = 0;        // SPEC
  int64_t off = 0;     // MEM / PARAM byte offset
  std::string label;   // LABEL
};

struct Inst {
  int line = 0;
  Kind k = K_RET;
  Ty ty = TY_NONE;   // operation type (destination type for cvt)
  Ty sty = TY_NONE;  // cvt source type
  Cmp cmp = C_EQ;
  Rnd rnd = R_NONE;
  int guard = -1;
  bool guard_neg = false;
  Opnd d, a, b, c;   // st: a = address, b = data; ld: a = address
  int target = -1;   // bra
  int event = -1;    // trace pseudo-op id
  int cls = ORC_LAT_ALU;
};

struct Param { std::string name; Ty ty; uint32_t off, size; };
struct Reg { std::string name; int width; };

struct Kernel {
  std::string name;
  std::vector<Param> params;
  uint32_t param_bytes = 0;
  std::vector<Reg> regs;
  std::map<std::string, int> reg_id;
  std::vector<Inst> code;
  std::vector<uint32_t> event_kind;   // 0 mark, 1 range_start, 2 range_end
  std::vector<std::string> event_name;
  std::vector<uint32_t> event_payload;  // payload bytes of each event: 0, 4 or 8
  // IKET NativeDump record size of the kernel's slots: 4 without payloads,
  // 4 + 4 with 4-byte payloads, 16 with 8-byte ones (the largest event's)
  uint32_t record_bytes = 4;
  std::vector<int> ipdom;             // per entry, n = virtual exit
  std::map<std::string, uint32_t> shared_sym;  // .shared array -> its shared address
  uint32_t shared_bytes = 0;
  bool has_bar = false;
  // CTA by CTA: the warps of a CTA share memory or barriers
  bool cta_mode() const { return shared_bytes > 0 || has_bar; }
};

// --------------------------------------------------------------- parsing ----
// Line-oriented preprocessing, then statements split on ';' inside the
// kernel body. Deliberately simple and separate from the library's lexer.

std::string trim(const std::string& s) {
  size_t a = 0, b = s.size();
  while (a < b && std::isspace((unsigned char)s[a])) a++;
  while (b > a && std::isspace((unsigned char)s[b - 1])) b--;
  return s.substr(a, b - a);
}

std::vector<std::string> split(const std::string& s, char sep) {
  std::vector<std::string> out;
  std::string cur;
  for (char ch : s) {
    if (ch == sep) { out.push_back(cur); cur.clear(); } else cur += ch;
  }
  out.push_back(cur);
  return out;
}

bool valid_ident(const std::string& s) {
  if (s.empty()) return false;
  char c0 = s[0];
  if (!(std::isalpha((unsigned char)c0) || c0 == '_' || c0 == '$')) return false;
  for (char ch : s) if (!(std::isalnum((unsigned char)ch) || ch == '_' || ch == '$')) return false;
  return true;
}

// One piece of source text with the line it started on.
struct Piece { std::string text; int line; };

// Removes comments, turns `//@iket kind name` into a statement `@iket kind name;`
// and drops .loc/.file lines. Keeps newlines so line numbers survive.
std::string preprocess(const std::string& src_in) {
  std::string src = src_in;
  for (char& ch : src) if (ch == '\t' || ch == '\r') ch = ' ';
  std::string nob;  // without block comments
  for (size_t i = 0; i < src.size();) {
    if (src.compare(i, 2, "/*") == 0) {
      size_t e = src.find("*/", i + 2);
      if (e == std::string::npos) fail(ORC_ERR_PARSE, 0, "unterminated block comment");
      for (size_t j = i; j < e + 2; j++) if (src[j] == '\n') nob += '\n';
      i = e + 2;
    } else {
      nob += src[i++];
    }
  }
  std::string out;
  std::vector<std::string> lines = split(nob, '\n');
  for (size_t li = 0; li < lines.size(); li++) {
    std::string line = lines[li];
    size_t cpos = line.find("//");
    std::string extra;
    if (cpos != std::string::npos) {
      std::string comment = line.substr(cpos + 2);
      line = line.substr(0, cpos);
      std::string ct = trim(comment);
      if (ct.compare(0, 5, "@iket") == 0) extra = " " + ct + ";";
    }
    std::string t = trim(line);
    if (t.compare(0, 4, ".loc") == 0 || t.compare(0, 5, ".file") == 0) line.clear();
    out += line + extra;
    if (li + 1 < lines.size()) out += '\n';
  }
  return out;
}

int line_of(const std::string& s, size_t pos) {
  int n = 1;
  for (size_t i = 0; i < pos && i < s.size(); i++) if (s[i] == '\n') n++;
  return n;
}

struct Lit { bool ok; bool neg; uint64_t mag; };

Lit parse_int_literal(std::string s) {
  Lit r{false, false, 0};
  if (s.empty()) return r;
  if (s[0] == '-') { r.neg = true; s = s.substr(1); }
  if (!s.empty() && (s.back() == 'U' || s.back() == 'u')) s.pop_back();
  if (s.empty()) return r;
  uint64_t v = 0;
  if (s.size() > 2 && s[0] == '0' && (s[1] == 'x' || s[1] == 'X')) {
    if (s.size() > 18) return r;
    for (size_t i = 2; i < s.size(); i++) {
      char ch = (char)std::tolower((unsigned char)s[i]);
      int dgt;
      if (ch >= '0' && ch <= '9') dgt = ch - '0';
      else if (ch >= 'a' && ch <= 'f') dgt = ch - 'a' + 10;
      else return r;
      v = v * 16 + (uint64_t)dgt;
    }
  } else {
    for (char ch : s) {
      if (ch < '0' || ch > '9') return r;
      uint64_t dgt = (uint64_t)(ch - '0');
      if (v > (UINT64_MAX - dgt) / 10) return r;
      v = v * 10 + dgt;
    }
  }
  r.ok = true;
  r.mag = v;
  return r;
}

bool parse_f32_literal(const std::string& s, uint64_t* bits) {
  if (s.size() != 10 || s[0] != '0' || (s[1] != 'f' && s[1] != 'F')) return false;
  uint64_t v = 0;
  for (size_t i = 2; i < 10; i++) {
    char ch = (char)std::tolower((unsigned char)s[i]);
    if (ch >= '0' && ch <= '9') v = v * 16 + (uint64_t)(ch - '0');
    else if (ch >= 'a' && ch <= 'f') v = v * 16 + (uint64_t)(ch - 'a' + 10);
    else return false;
  }
  *bits = v;
  return true;
}

struct Parser {
  Kernel& K;
  std::map<std::string, int> labels;        // label -> entry index
  std::vector<std::string> pending_labels;  // labels waiting for the next entry
  std::map<std::pair<uint32_t, std::string>, int> event_ids;

  explicit Parser(Kernel& k) : K(k) {}

  int reg_of(const std::string& name, int line) {
    auto it = K.reg_id.find(name);
    if (it == K.reg_id.end()) fail(ORC_ERR_PARSE, line, "undeclared register " + name);
    return it->second;
  }

  void declare_regs(const std::string& stmt, int line) {
    // .reg .TYPE %a<N>, %b, ...
    std::string rest = trim(stmt.substr(4));
    if (rest.empty() || rest[0] != '.') fail(ORC_ERR_PARSE, line, "bad .reg");
    size_t sp = 0;
    while (sp < rest.size() && !std::isspace((unsigned char)rest[sp])) sp++;
    Ty t = type_from(rest.substr(1, sp - 1));
    if (t == TY_NONE) fail(ORC_ERR_UNSUPPORTED, line, "unsupported register type " + rest.substr(0, sp));
    for (std::string nm : split(rest.substr(sp), ',')) {
      nm = trim(nm);
      if (nm.empty() || nm[0] != '%') fail(ORC_ERR_PARSE, line, "bad register name in .reg");
      size_t lt = nm.find('<');
      std::vector<std::string> names;
      if (lt == std::string::npos) {
        names.push_back(nm);
      } else {
        if (nm.back() != '>') fail(ORC_ERR_PARSE, line, "bad register range");
        Lit n = parse_int_literal(nm.substr(lt + 1, nm.size() - lt - 2));
        if (!n.ok || n.neg || n.mag == 0 || n.mag > 4096) fail(ORC_ERR_PARSE, line, "bad register count");
        std::string base = nm.substr(0, lt);
        for (uint64_t i = 0; i < n.mag; i++) names.push_back(base + std::to_string(i));
      }
      for (const std::string& r : names) {
        if (!valid_ident(r.substr(1))) fail(ORC_ERR_PARSE, line, "bad register name " + r);
        if (K.reg_id.count(r)) fail(ORC_ERR_PARSE, line, "register declared twice: " + r);
        K.reg_id[r] = (int)K.regs.size();
        K.regs.push_back(Reg{r, width_of(t)});
      }
    }
  }

  // .shared [.align A] .TYPE name[N]  (or a scalar without [N])
  void declare_shared(const std::string& stmt, int line) {
    std::vector<std::string> w;
    for (const std::string& x : split(stmt, ' '))
      for (const std::string& y : split(x, '\t'))
        if (!trim(y).empty()) w.push_back(trim(y));
    size_t i = 1;
    uint64_t align = 0;
    if (i + 1 < w.size() && w[i] == ".align") {
      Lit a = parse_int_literal(w[i + 1]);
      if (!a.ok || a.neg || a.mag == 0 || (a.mag & (a.mag - 1)) || a.mag > 4096) fail(ORC_ERR_PARSE, line, "bad .align");
      align = a.mag;
      i += 2;
    }
    if (i + 2 != w.size()) fail(ORC_ERR_UNSUPPORTED, line, "unsupported .shared declaration");
    static const std::map<std::string, uint32_t> esz = {
        {".b8", 1}, {".u8", 1}, {".s8", 1}, {".b16", 2}, {".u16", 2}, {".s16", 2},
        {".b32", 4}, {".u32", 4}, {".s32", 4}, {".f32", 4},
        {".b64", 8}, {".u64", 8}, {".s64", 8}, {".f64", 8}};
    auto et = esz.find(w[i]);
    if (et == esz.end()) fail(ORC_ERR_UNSUPPORTED, line, "unsupported .shared type " + w[i]);
    std::string nm = w[i + 1];
    uint64_t count = 1;
    size_t lb = nm.find('[');
    if (lb != std::string::npos) {
      if (nm.back() != ']') fail(ORC_ERR_PARSE, line, "bad .shared array");
      Lit c = parse_int_literal(nm.substr(lb + 1, nm.size() - lb - 2));
      if (!c.ok || c.neg || c.mag == 0 || c.mag > (1u << 20)) fail(ORC_ERR_PARSE, line, "bad .shared array size");
      count = c.mag;
      nm = nm.substr(0, lb);
    }
    if (!valid_ident(nm)) fail(ORC_ERR_PARSE, line, "bad .shared name");
    if (K.shared_sym.count(nm)) fail(ORC_ERR_PARSE, line, "shared array declared twice: " + nm);
    if (!align) align = et->second;
    const uint64_t off = (K.shared_bytes + align - 1) / align * align;
    const uint64_t end = off + count * et->second;
    if (end > 49152) fail(ORC_ERR_UNSUPPORTED, line, "more than 48 KiB of shared memory");
    K.shared_sym[nm] = (uint32_t)off;
    K.shared_bytes = (uint32_t)end;
  }

  // A shared address operand: [%r(+off)] with a 32- or 64-bit register, or
  // [symbol(+off)], which becomes a register-free address.
  void shared_address(Opnd& o, int line) {
    if (o.k == Opnd::PARAM) {
      auto it = K.shared_sym.find(o.label);
      if (it == K.shared_sym.end()) fail(ORC_ERR_PARSE, line, "unknown shared array " + o.label);
      o.k = Opnd::MEM;
      o.reg = -1;
      o.off += (int64_t)it->second;
      return;
    }
    if (o.k != Opnd::MEM || !(K.regs[o.reg].width == 32 || K.regs[o.reg].width == 64))
      fail(ORC_ERR_PARSE, line, "shared address must be [register(+offset)] or [array(+offset)]");
  }

  void add_entry(Inst in) {
    for (const std::string& l : pending_labels) labels[l] = (int)K.code.size();
    pending_labels.clear();
    K.code.push_back(in);
  }

  Opnd parse_operand(const std::string& raw, int line) {
    std::string s = trim(raw);
    Opnd o;
    if (s.empty()) fail(ORC_ERR_PARSE, line, "empty operand");
    if (s[0] == '[') {
      if (s.back() != ']') fail(ORC_ERR_PARSE, line, "bad address operand " + s);
      std::string in = trim(s.substr(1, s.size() - 2));
      std::string base = in, offs;
      int sign = 1;
      size_t p = in.find_first_of("+-", 1);
      if (p != std::string::npos) {
        base = trim(in.substr(0, p));
        sign = in[p] == '-' ? -1 : 1;
        offs = trim(in.substr(p + 1));
        if (!offs.empty() && offs[0] == '-') { sign = -sign; offs = trim(offs.substr(1)); }
        if (offs.empty()) fail(ORC_ERR_PARSE, line, "bad address offset");
      }
      int64_t off = 0;
      if (!offs.empty()) {
        Lit l = parse_int_literal(offs);
        if (!l.ok || l.neg || l.mag > 0x7FFFFFFFull) fail(ORC_ERR_PARSE, line, "bad address offset " + offs);
        off = sign * (int64_t)l.mag;
      }
      if (!base.empty() && base[0] == '%') {
        o.k = Opnd::MEM;
        o.reg = reg_of(base, line);
      } else {
        o.k = Opnd::PARAM;
        o.label = base;
      }
      o.off = off;
      return o;
    }
    if (s[0] == '%') {
      static const std::map<std::string, int> specials = {
          {"%tid.x", SP_TID_X}, {"%tid.y", SP_TID_Y}, {"%tid.z", SP_TID_Z},
          {"%ntid.x", SP_NTID_X}, {"%ntid.y", SP_NTID_Y}, {"%ntid.z", SP_NTID_Z},
          {"%ctaid.x", SP_CTAID_X}, {"%ctaid.y", SP_CTAID_Y}, {"%ctaid.z", SP_CTAID_Z},
          {"%nctaid.x", SP_NCTAID_X}, {"%nctaid.y", SP_NCTAID_Y}, {"%nctaid.z", SP_NCTAID_Z},
          {"%laneid", SP_LANEID}};
      auto it = specials.find(s);
      if (it != specials.end()) { o.k = Opnd::SPEC; o.spec = it->second; return o; }
      o.k = Opnd::REG;
      o.reg = reg_of(s, line);
      return o;
    }
    uint64_t fb;
    if (parse_f32_literal(s, &fb)) { o.k = Opnd::IMM; o.imm = fb; o.spec = 1; /* f32 literal */ return o; }
    if (std::isdigit((unsigned char)s[0]) || s[0] == '-') {
      Lit l = parse_int_literal(s);
      if (!l.ok) fail(ORC_ERR_PARSE, line, "bad literal " + s);
      o.k = Opnd::IMM;
      o.imm = l.neg ? (uint64_t)(0 - l.mag) : l.mag;
      o.spec = l.neg ? 3 : 2;  // 2 = non-negative int literal, 3 = negative
      o.off = (int64_t)l.mag;  // magnitude kept for range checks
      return o;
    }
    if (valid_ident(s)) { o.k = Opnd::LABEL; o.label = s; return o; }
    fail(ORC_ERR_PARSE, line, "bad operand " + s);
  }

  // Checks an operand against the width its position expects and truncates
  // immediates. kinds: 'r' register only, 'v' register or immediate,
  // 'm' register, immediate or special register, 'p' predicate register.
  void check(Opnd& o, int width, char kind, Ty ty, int line) {
    if (kind == 'p') {
      if (o.k != Opnd::REG || K.regs[o.reg].width != 1) fail(ORC_ERR_PARSE, line, "predicate register expected");
      return;
    }
    if (o.k == Opnd::REG) {
      if (K.regs[o.reg].width != width) fail(ORC_ERR_PARSE, line, "register width does not match the instruction type");
      return;
    }
    if (o.k == Opnd::SPEC) {
      if (kind != 'm' || width != 32) fail(ORC_ERR_PARSE, line, "special register only allowed as a 32-bit mov source");
      return;
    }
    if (o.k == Opnd::IMM) {
      if (kind == 'r') fail(ORC_ERR_PARSE, line, "register operand expected");
      bool f32lit = (o.spec == 1);
      if (f32lit) {
        if (!(ty == TY_F32 || ty == TY_B32)) fail(ORC_ERR_PARSE, line, "f32 literal on a non-32-bit-float operand");
      } else {
        if (ty == TY_F32) fail(ORC_ERR_PARSE, line, "f32 operands take 0fXXXXXXXX literals only");
        uint64_t mag = (uint64_t)o.off;
        bool neg = (o.spec == 3);
        if (width == 32) {
          if (neg ? mag > 0x80000000ull : mag > 0xFFFFFFFFull) fail(ORC_ERR_PARSE, line, "literal does not fit 32 bits");
          o.imm &= 0xFFFFFFFFull;
        } else if (neg && mag > 0x8000000000000000ull) {
          fail(ORC_ERR_PARSE, line, "literal does not fit 64 bits");
        }
      }
      return;
    }
    fail(ORC_ERR_PARSE, line, "bad operand kind");
  }

  void instruction(const std::string& stmt, int line) {
    Inst in;
    in.line = line;
    std::string s = stmt;
    if (s[0] == '@') {
      size_t sp = 0;
      while (sp < s.size() && !std::isspace((unsigned char)s[sp])) sp++;
      std::string g = s.substr(1, sp - 1);
      if (!g.empty() && g[0] == '!') { in.guard_neg = true; g = g.substr(1); }
      if (g.empty() || g[0] != '%') fail(ORC_ERR_PARSE, line, "bad guard");
      in.guard = reg_of(g, line);
      if (K.regs[in.guard].width != 1) fail(ORC_ERR_PARSE, line, "guard must be a predicate");
      s = trim(s.substr(sp));
    }
    size_t sp = 0;
    while (sp < s.size() && !std::isspace((unsigned char)s[sp])) sp++;
    std::vector<std::string> parts = split(s.substr(0, sp), '.');
    std::string op = parts[0];
    std::vector<std::string> mods(parts.begin() + 1, parts.end());
    std::string rest = trim(s.substr(sp));
    std::vector<Opnd> ops;
    if (!rest.empty())
      for (const std::string& p : split(rest, ',')) ops.push_back(parse_operand(p, line));
    auto need = [&](size_t n) {
      if (ops.size() != n) fail(ORC_ERR_PARSE, line, op + ": expected " + std::to_string(n) + " operands");
    };
    auto bad = [&]() { fail(ORC_ERR_UNSUPPORTED, line, "unsupported instruction form: " + s.substr(0, sp)); };

    if (op == "add" || op == "sub" || op == "mul" || op == "mad" || op == "fma" || op == "div" ||
        op == "sqrt") {
      bool rn = false, lo = false;
      Ty t = TY_NONE;
      for (const std::string& m : mods) {
        if (m == "rn" && !rn) rn = true;
        else if (m == "lo" && !lo) lo = true;
        else if (t == TY_NONE && type_from(m) != TY_NONE) t = type_from(m);
        else bad();
      }
      if (t == TY_NONE) bad();
      in.ty = t;
      if (op == "add" || op == "sub") {
        in.k = op == "add" ? K_ADD : K_SUB;
        if (lo) bad();
        if (t == TY_F32) { /* .rn optional */ } else if (!is_int_ty(t) || rn) bad();
        need(3);
      } else if (op == "mul") {
        in.k = K_MUL;
        if (t == TY_F32) { if (lo) bad(); } else if (!is_int_ty(t) || !lo || rn) bad();
        need(3);
      } else if (op == "mad") {
        in.k = K_MAD;
        if (!is_int_ty(t) || !lo || rn) bad();
        need(4);
      } else if (op == "fma") {
        in.k = K_FMA;
        if (t != TY_F32 || !rn || lo) bad();
        need(4);
        in.cls = ORC_LAT_FMA;
      } else if (op == "div") {
        in.k = K_DIV;
        if (t != TY_F32 || !rn || lo) bad();
        need(3);
        in.cls = ORC_LAT_SFU;
      } else {
        in.k = K_SQRT;
        if (t != TY_F32 || !rn || lo) bad();
        need(2);
        in.cls = ORC_LAT_SFU;
      }
      int w = width_of(t);
      in.d = ops[0]; check(in.d, w, 'r', t, line);
      in.a = ops[1]; check(in.a, w, 'v', t, line);
      if (ops.size() > 2) { in.b = ops[2]; check(in.b, w, 'v', t, line); }
      if (ops.size() > 3) { in.c = ops[3]; check(in.c, w, 'v', t, line); }
    } else if (op == "and" || op == "or" || op == "xor") {
      in.k = op == "and" ? K_AND : (op == "or" ? K_OR : K_XOR);
      if (mods.size() != 1) bad();
      Ty t = type_from(mods[0]);
      if (!(t == TY_B32 || t == TY_B64 || t == TY_PRED)) bad();
      in.ty = t;
      need(3);
      in.d = ops[0]; in.a = ops[1]; in.b = ops[2];
      if (t == TY_PRED) {
        check(in.d, 1, 'p', t, line); check(in.a, 1, 'p', t, line); check(in.b, 1, 'p', t, line);
      } else {
        int w = width_of(t);
        check(in.d, w, 'r', t, line); check(in.a, w, 'v', t, line); check(in.b, w, 'v', t, line);
      }
    } else if (op == "shl" || op == "shr") {
      in.k = op == "shl" ? K_SHL : K_SHR;
      if (mods.size() != 1) bad();
      Ty t = type_from(mods[0]);
      if (op == "shl" && !(t == TY_B32 || t == TY_B64)) bad();
      if (op == "shr" && !(t == TY_B32 || t == TY_B64 || is_int_ty(t))) bad();
      in.ty = t;
      need(3);
      int w = width_of(t);
      in.d = ops[0]; check(in.d, w, 'r', t, line);
      in.a = ops[1]; check(in.a, w, 'v', t, line);
      in.b = ops[2]; check(in.b, 32, 'v', TY_U32, line);
    } else if (op == "cvt") {
      in.k = K_CVT;
      std::vector<std::string> m = mods;
      Rnd r = R_NONE;
      if (!m.empty()) {
        if (m[0] == "rn") r = R_RN;
        else if (m[0] == "rni") r = R_RNI;
        else if (m[0] == "rzi") r = R_RZI;
        else if (m[0] == "rmi") r = R_RMI;
        else if (m[0] == "rpi") r = R_RPI;
        if (r != R_NONE) m.erase(m.begin());
      }
      if (m.size() != 2) bad();
      Ty dt = type_from(m[0]), st = type_from(m[1]);
      if (is_int_ty(dt) && is_int_ty(st)) { if (r != R_NONE) bad(); }
      else if (dt == TY_F32 && is_int_ty(st)) { if (r != R_RN) bad(); }
      else if (is_int_ty(dt) && st == TY_F32) { if (r == R_NONE || r == R_RN) bad(); }
      else bad();
      in.ty = dt; in.sty = st; in.rnd = r;
      need(2);
      in.d = ops[0]; check(in.d, width_of(dt), 'r', dt, line);
      in.a = ops[1]; check(in.a, width_of(st), 'r', st, line);
    } else if (op == "mov") {
      in.k = K_MOV;
      if (mods.size() != 1) bad();
      Ty t = type_from(mods[0]);
      if (t == TY_NONE || t == TY_PRED) bad();
      in.ty = t;
      need(2);
      int w = width_of(t);
      in.d = ops[0]; check(in.d, w, 'r', t, line);
      in.a = ops[1];
      if (in.a.k == Opnd::LABEL) {  // the shared address of an array
        auto it = K.shared_sym.find(in.a.label);
        if (it == K.shared_sym.end() || t == TY_F32) fail(ORC_ERR_PARSE, line, "bad mov operand " + in.a.label);
        in.a.k = Opnd::IMM;
        in.a.imm = it->second;
        in.a.spec = 2;
        in.a.off = it->second;
      }
      check(in.a, w, 'm', t, line);
    } else if (op == "setp") {
      in.k = K_SETP;
      if (mods.size() != 2) bad();
      Ty t = type_from(mods[1]);
      const std::string& c = mods[0];
      bool uns_name = (c == "lo" || c == "ls" || c == "hi" || c == "hs");
      if (c == "eq") in.cmp = C_EQ; else if (c == "ne") in.cmp = C_NE;
      else if (c == "lt" || c == "lo") in.cmp = C_LT; else if (c == "le" || c == "ls") in.cmp = C_LE;
      else if (c == "gt" || c == "hi") in.cmp = C_GT; else if (c == "ge" || c == "hs") in.cmp = C_GE;
      else bad();
      if (t == TY_B32 || t == TY_B64) { if (!(in.cmp == C_EQ || in.cmp == C_NE)) bad(); }
      else if (t == TY_U32 || t == TY_U64) { }
      else if (t == TY_S32 || t == TY_S64 || t == TY_F32) { if (uns_name) bad(); }
      else bad();
      in.ty = t;
      need(3);
      int w = width_of(t);
      in.d = ops[0]; check(in.d, 1, 'p', t, line);
      in.a = ops[1]; check(in.a, w, 'v', t, line);
      in.b = ops[2]; check(in.b, w, 'v', t, line);
    } else if (op == "selp") {
      in.k = K_SELP;
      if (mods.size() != 1) bad();
      Ty t = type_from(mods[0]);
      if (t == TY_NONE || t == TY_PRED) bad();
      in.ty = t;
      need(4);
      int w = width_of(t);
      in.d = ops[0]; check(in.d, w, 'r', t, line);
      in.a = ops[1]; check(in.a, w, 'v', t, line);
      in.b = ops[2]; check(in.b, w, 'v', t, line);
      in.c = ops[3]; check(in.c, 1, 'p', t, line);
    } else if (op == "bra") {
      in.k = K_BRA;
      in.cls = ORC_LAT_BRA;
      if (!(mods.empty() || (mods.size() == 1 && mods[0] == "uni"))) bad();
      need(1);
      if (ops[0].k != Opnd::LABEL) fail(ORC_ERR_PARSE, line, "bra needs a label");
      in.a = ops[0];
    } else if (op == "bar" || op == "barrier") {
      // bar.sync 0 / barrier.sync[.aligned] 0: CTA barrier 0 over every thread
      const bool form = (op == "bar" && mods.size() == 1 && mods[0] == "sync") ||
                        (op == "barrier" && (mods.size() == 1 || mods.size() == 2) && mods[0] == "sync" &&
                         (mods.size() == 1 || mods[1] == "aligned"));
      if (!form) bad();
      need(1);
      if (ops[0].k != Opnd::IMM || ops[0].spec != 2 || ops[0].imm != 0)
        fail(ORC_ERR_UNSUPPORTED, line, "only barrier 0 without a thread count is supported");
      if (in.guard >= 0) fail(ORC_ERR_UNSUPPORTED, line, "guarded bar.sync is not supported");
      in.k = K_BAR;
      in.cls = ORC_LAT_BAR;
      K.has_bar = true;
    } else if (op == "ret" || op == "exit") {
      in.k = K_RET;
      in.cls = ORC_LAT_RET;
      if (!mods.empty()) bad();
      need(0);
    } else if (op == "ld" || op == "st") {
      if (mods.size() != 2) bad();
      Ty t = type_from(mods[1]);
      if (t == TY_NONE || t == TY_PRED) bad();
      in.ty = t;
      int w = width_of(t);
      need(2);
      if (op == "ld" && mods[0] == "global") {
        in.k = K_LDG; in.cls = ORC_LAT_LDG;
        in.d = ops[0]; check(in.d, w, 'r', t, line);
        in.a = ops[1];
        if (in.a.k != Opnd::MEM || K.regs[in.a.reg].width != 64) fail(ORC_ERR_PARSE, line, "ld.global needs [64-bit register(+offset)]");
      } else if (op == "ld" && mods[0] == "param") {
        in.k = K_LDP;
        in.d = ops[0]; check(in.d, w, 'r', t, line);
        in.a = ops[1];
        if (in.a.k != Opnd::PARAM) fail(ORC_ERR_PARSE, line, "ld.param needs [param(+offset)]");
        const Param* pp = nullptr;
        for (const Param& p : K.params) if (p.name == in.a.label) pp = &p;
        if (!pp) fail(ORC_ERR_PARSE, line, "unknown parameter " + in.a.label);
        int64_t addr = (int64_t)pp->off + in.a.off;
        int64_t size = w / 8;
        if (addr < 0 || addr + size > (int64_t)K.param_bytes || addr % size != 0)
          fail(ORC_ERR_PARSE, line, "ld.param outside the parameter block or misaligned");
        in.a.off = addr;
      } else if (op == "st" && mods[0] == "global") {
        in.k = K_STG; in.cls = ORC_LAT_STG;
        in.a = ops[0];
        if (in.a.k != Opnd::MEM || K.regs[in.a.reg].width != 64) fail(ORC_ERR_PARSE, line, "st.global needs [64-bit register(+offset)]");
        in.b = ops[1]; check(in.b, w, 'r', t, line);
      } else if (op == "ld" && mods[0] == "shared") {
        in.k = K_LDS; in.cls = ORC_LAT_LDS;
        in.d = ops[0]; check(in.d, w, 'r', t, line);
        in.a = ops[1]; shared_address(in.a, line);
      } else if (op == "st" && mods[0] == "shared") {
        in.k = K_STS; in.cls = ORC_LAT_STS;
        in.a = ops[0]; shared_address(in.a, line);
        in.b = ops[1]; check(in.b, w, 'r', t, line);
      } else {
        bad();
      }
    } else {
      fail(ORC_ERR_UNSUPPORTED, line, "unsupported opcode " + op);
    }
    add_entry(in);
  }

  // `@iket KIND NAME [%reg]`: an optional payload register (its value in the
  // warp's lowest active lane goes into the record)
  void event(const std::string& stmt, int line) {
    std::vector<std::string> w;
    for (const std::string& t : split(stmt, ' ')) if (!trim(t).empty()) w.push_back(trim(t));
    if (w.size() != 3 && w.size() != 4) fail(ORC_ERR_PARSE, line, "bad //@iket pseudo-op");
    int preg = -1;
    uint32_t pbytes = 0;
    if (w.size() == 4) {
      if (w[3].empty() || w[3][0] != '%') fail(ORC_ERR_PARSE, line, "an //@iket payload must be a register");
      preg = reg_of(w[3], line);
      const int pw = K.regs[(size_t)preg].width;
      if (pw != 32 && pw != 64) fail(ORC_ERR_PARSE, line, "an //@iket payload must be a 32- or 64-bit register");
      pbytes = (uint32_t)pw / 8;
    }
    uint32_t kind;
    if (w[1] == "mark") kind = 0;
    else if (w[1] == "range_start") kind = 1;
    else if (w[1] == "range_end") kind = 2;
    else fail(ORC_ERR_PARSE, line, "unknown //@iket kind " + w[1]);
    if (!valid_ident(w[2])) fail(ORC_ERR_PARSE, line, "bad event name");
    auto key = std::make_pair(kind, w[2]);
    auto it = event_ids.find(key);
    int id;
    if (it == event_ids.end()) {
      id = (int)K.event_kind.size();
      if (id >= 256) fail(ORC_ERR_UNSUPPORTED, line, "more than 256 events");
      event_ids[key] = id;
      K.event_kind.push_back(kind);
      K.event_name.push_back(w[2]);
      K.event_payload.push_back(pbytes);
    } else {
      id = it->second;
      if (K.event_payload[(size_t)id] != pbytes)
        fail(ORC_ERR_PARSE, line, "event " + w[2] + " used with two payload sizes");
    }
    K.record_bytes = std::max(K.record_bytes, pbytes == 0 ? 4u : pbytes == 4 ? 8u : 16u);
    Inst in;
    in.line = line;
    in.k = K_EVENT;
    in.event = id;
    if (preg >= 0) { in.a.k = Opnd::REG; in.a.reg = preg; }
    add_entry(in);
  }

  void statement(std::string s, int line) {
    s = trim(s);
    // Leading labels.
    while (true) {
      size_t colon = s.find(':');
      if (colon == std::string::npos) break;
      std::string lab = trim(s.substr(0, colon));
      if (!valid_ident(lab)) break;
      if (labels.count(lab) || std::count(pending_labels.begin(), pending_labels.end(), lab))
        fail(ORC_ERR_PARSE, line, "label defined twice: " + lab);
      pending_labels.push_back(lab);
      s = trim(s.substr(colon + 1));
    }
    if (s.empty()) return;
    if (s.compare(0, 4, ".reg") == 0) { declare_regs(s, line); return; }
    if (s.compare(0, 7, ".shared") == 0) { declare_shared(s, line); return; }
    if (s.compare(0, 5, "@iket") == 0) { event(s, line); return; }
    if (s[0] == '.') fail(ORC_ERR_UNSUPPORTED, line, "unsupported directive in kernel body: " + s);
    instruction(s, line);
  }

  void finish() {
    if (!pending_labels.empty()) fail(ORC_ERR_PARSE, 0, "label at the end of the kernel: " + pending_labels[0]);
    if (K.code.empty()) fail(ORC_ERR_PARSE, 0, "empty kernel");
    for (Inst& in : K.code) {
      if (in.k != K_BRA) continue;
      auto it = labels.find(in.a.label);
      if (it == labels.end()) fail(ORC_ERR_PARSE, in.line, "undefined label " + in.a.label);
      in.target = it->second;
    }
    const Inst& last = K.code.back();
    if (!((last.k == K_RET || last.k == K_BRA) && last.guard < 0))
      fail(ORC_ERR_PARSE, last.line, "control can fall off the end of the kernel");
  }
};

void parse_params(Kernel& K, const std::string& text, int line) {
  std::string t = trim(text);
  if (t.empty()) return;
  uint32_t off = 0;
  for (std::string p : split(t, ',')) {
    p = trim(p);
    std::vector<std::string> w;
    for (const std::string& x : split(p, ' ')) {
      std::string y = trim(x);
      if (!y.empty()) for (const std::string& z : split(y, '\t')) if (!trim(z).empty()) w.push_back(trim(z));
    }
    if (w.size() != 3 || w[0] != ".param" || w[1].empty() || w[1][0] != '.')
      fail(ORC_ERR_UNSUPPORTED, line, "unsupported parameter declaration: " + p);
    Ty ty = type_from(w[1].substr(1));
    if (ty == TY_NONE || ty == TY_PRED) fail(ORC_ERR_UNSUPPORTED, line, "unsupported parameter type " + w[1]);
    if (!valid_ident(w[2])) fail(ORC_ERR_PARSE, line, "bad parameter name " + w[2]);
    for (const Param& q : K.params) if (q.name == w[2]) fail(ORC_ERR_PARSE, line, "parameter declared twice");
    uint32_t size = (uint32_t)width_of(ty) / 8;
    off = (off + size - 1) / size * size;  // natural alignment
    K.params.push_back(Param{w[2], ty, off, size});
    off += size;
  }
  K.param_bytes = off;
}

void compute_ipdom(Kernel& K);

// Parses the module and returns the requested kernel.
Kernel load(const std::string& src, const std::string& want) {
  std::string s = preprocess(src);
  size_t pos = 0;
  bool found = false;
  Kernel result;
  while (pos < s.size()) {
    while (pos < s.size() && std::isspace((unsigned char)s[pos])) pos++;
    if (pos >= s.size()) break;
    size_t e = pos;
    while (e < s.size() && !std::isspace((unsigned char)s[e]) && s[e] != '(') e++;
    std::string word = s.substr(pos, e - pos);
    int line = line_of(s, pos);
    if (word == ".version" || word == ".target") {
      size_t nl = s.find('\n', pos);
      pos = nl == std::string::npos ? s.size() : nl;
      continue;
    }
    if (word == ".address_size") {
      size_t nl = s.find('\n', pos);
      std::string v = trim(s.substr(e, (nl == std::string::npos ? s.size() : nl) - e));
      if (v != "64") fail(ORC_ERR_UNSUPPORTED, line, "only .address_size 64 is supported");
      pos = nl == std::string::npos ? s.size() : nl;
      continue;
    }
    if (word == ".visible") { pos = e; continue; }
    if (word != ".entry") fail(ORC_ERR_UNSUPPORTED, line, "unsupported top-level statement " + word);
    // .entry NAME ( params ) [directives] { body }
    size_t lp = s.find('(', e);
    if (lp == std::string::npos) fail(ORC_ERR_PARSE, line, "missing '(' after .entry");
    std::string name = trim(s.substr(e, lp - e));
    if (!valid_ident(name)) fail(ORC_ERR_PARSE, line, "bad kernel name");
    size_t rp = s.find(')', lp);
    if (rp == std::string::npos) fail(ORC_ERR_PARSE, line, "missing ')'");
    size_t lb = s.find('{', rp);
    if (lb == std::string::npos) fail(ORC_ERR_PARSE, line, "missing '{'");
    size_t rb = s.find('}', lb);
    if (rb == std::string::npos) fail(ORC_ERR_PARSE, line, "missing '}'");
    std::string body = s.substr(lb + 1, rb - lb - 1);
    if (body.find('{') != std::string::npos) fail(ORC_ERR_UNSUPPORTED, line_of(s, lb), "nested blocks are not supported");
    if (name == want && !found) {
      found = true;
      result.name = name;
      parse_params(result, s.substr(lp + 1, rp - lp - 1), line);
      Parser P(result);
      size_t start = 0;
      int base_line = line_of(s, lb + 1);
      for (size_t i = 0; i <= body.size(); i++) {
        if (i == body.size() || body[i] == ';') {
          std::string piece = body.substr(start, i - start);
          // line of the first non-space character of the piece
          size_t k = 0;
          while (k < piece.size() && std::isspace((unsigned char)piece[k])) k++;
          int ln = base_line;
          for (size_t j = 0; j < start + k && j < body.size(); j++) if (body[j] == '\n') ln++;
          if (i == body.size()) {
            // trailing text without ';' may only be labels
            std::string t = trim(piece);
            if (!t.empty()) {
              if (t.back() != ':') fail(ORC_ERR_PARSE, ln, "missing ';'");
              P.statement(t, ln);
            }
          } else {
            P.statement(piece, ln);
          }
          start = i + 1;
        }
      }
      P.finish();
    }
    pos = rb + 1;
  }
  if (!found) throw OracleError{ORC_ERR_NOT_FOUND, "kernel not found: " + want};
  compute_ipdom(result);
  return result;
}

// ------------------------------------------------------ post-dominators ----
// Plain iterative post-dominator sets: pdom(exit) = {exit};
// pdom(n) = {n} ∪ ⋂ pdom(s) over successors s that can reach the exit.
// ipdom(n) is the strict post-dominator d with pdom(d) = pdom(n) \ {n}.
// Entries that cannot reach the exit reconverge at the virtual exit.

std::vector<int> successors(const Kernel& K, int i) {
  const Inst& in = K.code[(size_t)i];
  int n = (int)K.code.size();
  std::vector<int> s;
  if (in.k == K_BRA) {
    s.push_back(in.target);
    if (in.guard >= 0 && i + 1 != in.target) s.push_back(i + 1);
  } else if (in.k == K_RET) {
    s.push_back(n);
    if (in.guard >= 0) s.push_back(i + 1);
  } else {
    s.push_back(i + 1);
  }
  return s;
}

void compute_ipdom(Kernel& K) {
  int n = (int)K.code.size();
  std::vector<std::vector<int>> succ((size_t)n);
  for (int i = 0; i < n; i++) succ[(size_t)i] = successors(K, i);
  // which entries can reach the exit
  std::vector<bool> reach((size_t)n + 1, false);
  reach[(size_t)n] = true;
  bool changed = true;
  while (changed) {
    changed = false;
    for (int i = 0; i < n; i++) {
      if (reach[(size_t)i]) continue;
      for (int s : succ[(size_t)i]) if (reach[(size_t)s]) { reach[(size_t)i] = true; changed = true; break; }
    }
  }
  std::set<int> all;
  for (int i = 0; i <= n; i++) all.insert(i);
  std::vector<std::set<int>> pdom((size_t)n + 1, all);
  pdom[(size_t)n] = {n};
  changed = true;
  while (changed) {
    changed = false;
    for (int i = n - 1; i >= 0; i--) {
      if (!reach[(size_t)i]) continue;
      std::set<int> acc;
      bool first = true;
      for (int s : succ[(size_t)i]) {
        if (!reach[(size_t)s]) continue;
        if (first) { acc = pdom[(size_t)s]; first = false; }
        else {
          std::set<int> tmp;
          std::set_intersection(acc.begin(), acc.end(), pdom[(size_t)s].begin(), pdom[(size_t)s].end(),
                                std::inserter(tmp, tmp.begin()));
          acc = tmp;
        }
      }
      acc.insert(i);
      if (acc != pdom[(size_t)i]) { pdom[(size_t)i] = acc; changed = true; }
    }
  }
  K.ipdom.assign((size_t)n, n);
  for (int i = 0; i < n; i++) {
    if (!reach[(size_t)i]) continue;
    std::set<int> strict = pdom[(size_t)i];
    strict.erase(i);
    for (int d : strict) {
      if (pdom[(size_t)d] == strict) { K.ipdom[(size_t)i] = d; break; }
    }
  }
}

// -------------------------------------------------------------- memory ----

struct Memory {
  const orc_buffer* bufs;
  uint32_t n;
  // race checker state, one entry per 4-byte word of each buffer
  bool race_on = false;
  std::vector<std::vector<int64_t>> writer, reader;
  uint32_t race_flags = 0;

  // returns 0 and the host pointer, or a status code
  int translate(uint64_t addr, uint32_t size, uint8_t** host, int* buf_index, uint64_t* offset) const {
    if (addr % size != 0) return ORC_ST_MISALIGNED;
    for (uint32_t i = 0; i < n; i++) {
      const orc_buffer& b = bufs[i];
      if (addr >= b.sim_base && b.bytes >= size && addr - b.sim_base <= b.bytes - size) {
        *offset = addr - b.sim_base;
        *host = (uint8_t*)b.host + *offset;
        *buf_index = (int)i;
        return 0;
      }
    }
    return ORC_ST_OOB;
  }

  void note(int bi, uint64_t off, uint32_t size, int64_t gtid, bool write) {
    if (!race_on) return;
    for (uint64_t w = off / 4; w < (off + size) / 4; w++) {
      int64_t& wr = writer[(size_t)bi][(size_t)w];
      int64_t& rd = reader[(size_t)bi][(size_t)w];
      if (write) {
        if (wr >= 0 && wr != gtid) race_flags |= ORC_RACE_CROSS_THREAD;
        if (rd != -1 && rd != gtid) race_flags |= ORC_RACE_CROSS_THREAD;
        wr = gtid;
      } else {
        if (wr >= 0 && wr != gtid) race_flags |= ORC_RACE_CROSS_THREAD;
        if (rd == -1) rd = gtid; else if (rd != gtid) rd = -2;
      }
    }
  }
};

// ------------------------------------------------------------ semantics ----

uint64_t trunc_to(uint64_t v, int width) { return width == 64 ? v : (v & 0xFFFFFFFFull); }

int64_t as_signed(uint64_t v, int width) {
  if (width == 64) return (int64_t)v;
  return (int64_t)(int32_t)(uint32_t)v;
}

float to_f(uint64_t v) {
  uint32_t u = (uint32_t)v;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Result of an f32 arithmetic operation; NaN results are canonical.
uint64_t from_f(float f) {
  if (std::isnan(f)) return 0x7FFFFFFFull;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

// Float to integer: round to an integral value in the given direction,
// then saturate to the destination range; NaN gives 0.
uint64_t f2i(float f, Rnd r, Ty dt) {
  if (std::isnan(f)) return 0;
  float x;
  switch (r) {
    case R_RZI: x = std::trunc(f); break;
    case R_RMI: x = std::floor(f); break;
    case R_RPI: x = std::ceil(f); break;
    default: x = std::nearbyint(f); break;  // default rounding mode: nearest, ties to even
  }
  switch (dt) {
    case TY_S32:
      if (x >= 2147483648.0f) return 0x7FFFFFFFull;
      if (x < -2147483648.0f) return 0x80000000ull;
      return (uint64_t)(uint32_t)(int32_t)x;
    case TY_U32:
      if (x >= 4294967296.0f) return 0xFFFFFFFFull;
      if (x < 0.0f) return 0;
      return (uint64_t)(uint32_t)x;
    case TY_S64:
      if (x >= 9223372036854775808.0f) return 0x7FFFFFFFFFFFFFFFull;
      if (x < -9223372036854775808.0f) return 0x8000000000000000ull;
      return (uint64_t)(int64_t)x;
    default:  // u64
      if (x >= 18446744073709551616.0f) return 0xFFFFFFFFFFFFFFFFull;
      if (x < 0.0f) return 0;
      return (uint64_t)x;
  }
}

struct Lane {
  std::vector<uint64_t> v;  // one value per declared register (predicates 0/1)
};

struct LaneCtx { uint32_t tid, ntid, ctaid, nctaid, laneid; };

uint64_t special_value(int sp, const LaneCtx& c) {
  switch (sp) {
    case SP_TID_X: return c.tid;
    case SP_NTID_X: return c.ntid;
    case SP_CTAID_X: return c.ctaid;
    case SP_NCTAID_X: return c.nctaid;
    case SP_LANEID: return c.laneid;
    case SP_NTID_Y: case SP_NTID_Z: case SP_NCTAID_Y: case SP_NCTAID_Z: return 1;
    default: return 0;  // tid.y/z, ctaid.y/z
  }
}

uint64_t value(const Lane& L, const Opnd& o, int width, const LaneCtx& c) {
  if (o.k == Opnd::REG) return L.v[(size_t)o.reg];
  if (o.k == Opnd::IMM) return trunc_to(o.imm, width);
  return special_value(o.spec, c);
}

bool compare(Cmp cmp, Ty t, uint64_t a, uint64_t b) {
  if (t == TY_F32) {
    float x = to_f(a), y = to_f(b);
    if (std::isnan(x) || std::isnan(y)) return false;  // ordered comparisons
    switch (cmp) {
      case C_EQ: return x == y; case C_NE: return x != y; case C_LT: return x < y;
      case C_LE: return x <= y; case C_GT: return x > y; default: return x >= y;
    }
  }
  int w = width_of(t);
  if (is_signed_ty(t)) {
    int64_t x = as_signed(a, w), y = as_signed(b, w);
    switch (cmp) {
      case C_EQ: return x == y; case C_NE: return x != y; case C_LT: return x < y;
      case C_LE: return x <= y; case C_GT: return x > y; default: return x >= y;
    }
  }
  uint64_t x = trunc_to(a, w), y = trunc_to(b, w);
  switch (cmp) {
    case C_EQ: return x == y; case C_NE: return x != y; case C_LT: return x < y;
    case C_LE: return x <= y; case C_GT: return x > y; default: return x >= y;
  }
}

// Executes one non-control, non-memory instruction for one lane.
void alu(const Inst& in, Lane& L, const LaneCtx& c, const uint8_t* params) {
  int w = width_of(in.ty);
  uint64_t r = 0;
  switch (in.k) {
    case K_ADD: case K_SUB: case K_MUL: case K_MAD: {
      uint64_t a = value(L, in.a, w, c), b = value(L, in.b, w, c);
      if (in.ty == TY_F32) {
        float x = to_f(a), y = to_f(b);
        r = from_f(in.k == K_ADD ? x + y : in.k == K_SUB ? x - y : x * y);
      } else if (in.k == K_ADD) r = a + b;
      else if (in.k == K_SUB) r = a - b;
      else if (in.k == K_MUL) r = a * b;
      else r = a * b + value(L, in.c, w, c);
      break;
    }
    case K_FMA:
      r = from_f(std::fma(to_f(value(L, in.a, w, c)), to_f(value(L, in.b, w, c)), to_f(value(L, in.c, w, c))));
      break;
    case K_DIV: r = from_f(to_f(value(L, in.a, w, c)) / to_f(value(L, in.b, w, c))); break;
    case K_SQRT: r = from_f(std::sqrt(to_f(value(L, in.a, w, c)))); break;
    case K_AND: case K_OR: case K_XOR: {
      uint64_t a = value(L, in.a, w, c), b = value(L, in.b, w, c);
      r = in.k == K_AND ? (a & b) : in.k == K_OR ? (a | b) : (a ^ b);
      if (in.ty == TY_PRED) r &= 1;
      break;
    }
    case K_SHL: case K_SHR: {
      uint64_t a = value(L, in.a, w, c);
      uint64_t amt = value(L, in.b, 32, c);
      if (in.k == K_SHL) r = amt >= (uint64_t)w ? 0 : (a << amt);
      else if (is_signed_ty(in.ty)) {
        int64_t sa = as_signed(a, w);
        r = (uint64_t)(amt >= (uint64_t)w ? (sa < 0 ? -1 : 0) : (sa >> amt));
      } else r = amt >= (uint64_t)w ? 0 : (trunc_to(a, w) >> amt);
      break;
    }
    case K_CVT: {
      int sw = width_of(in.sty);
      uint64_t a = value(L, in.a, sw, c);
      if (in.sty == TY_F32) r = f2i(to_f(a), in.rnd, in.ty);
      else if (in.ty == TY_F32) {
        float f;
        if (in.sty == TY_U32) f = (float)(uint32_t)a;
        else if (in.sty == TY_S32) f = (float)(int32_t)(uint32_t)a;
        else if (in.sty == TY_U64) f = (float)a;
        else f = (float)(int64_t)a;
        uint32_t u;
        std::memcpy(&u, &f, 4);
        r = u;
      } else {
        r = is_signed_ty(in.sty) ? (uint64_t)as_signed(a, sw) : trunc_to(a, sw);
      }
      break;
    }
    case K_MOV: r = value(L, in.a, w, c); break;
    case K_SETP: r = compare(in.cmp, in.ty, value(L, in.a, w, c), value(L, in.b, w, c)) ? 1 : 0; break;
    case K_SELP: r = L.v[(size_t)in.c.reg] ? value(L, in.a, w, c) : value(L, in.b, w, c); break;
    case K_LDP: {
      r = 0;
      for (int i = w / 8 - 1; i >= 0; i--) r = (r << 8) | params[in.a.off + i];
      break;
    }
    default: break;
  }
  int dw = (in.k == K_SETP) ? 1 : w;
  L.v[(size_t)in.d.reg] = dw == 1 ? (r & 1) : trunc_to(r, dw);
}

uint64_t load_le(const uint8_t* p, uint32_t size) {
  uint64_t r = 0;
  for (int i = (int)size - 1; i >= 0; i--) r = (r << 8) | p[i];
  return r;
}

void store_le(uint8_t* p, uint64_t v, uint32_t size) {
  for (uint32_t i = 0; i < size; i++) { p[i] = (uint8_t)(v & 0xFF); v >>= 8; }
}

int popcount32(uint32_t m) {
  int n = 0;
  for (int i = 0; i < 32; i++) n += (m >> i) & 1;
  return n;
}

struct CacheModel;

// One event of the kind the page's hints analyzer reads: a global request
// (a = executing lanes, b = distinct lines, c = access bytes), a shared
// request (a = bank-conflict degree), a divergent branch (a = taken lanes,
// b = fall-through lanes).
struct HintEvent { uint32_t pc, kind, a, b, c, pad; };
enum { EV_GLOBAL = 0, EV_SHARED = 1, EV_DIVERGE = 2 };

struct Launch {
  const Kernel* K;
  uint32_t grid, block, warps_per_cta;
  const uint8_t* params;
  const orc_config* cfg;
  uint8_t* stats;
  uint8_t* trace;
  uint64_t slot_bytes;
  CacheModel* cache = nullptr;  // L1/L2 hit model, or none
  uint8_t* cache_warps = nullptr;  // W x {u32 n_access, l1_hits, l2_hits, dram}
  uint8_t* cache_log = nullptr;    // W x cache_cap x {u64 line, u32 step, u32 level}
  uint32_t cache_cap = 0;
  std::vector<HintEvent>* events = nullptr;  // hint events, in run order (one host thread)
};

// ------------------------------------------------------- L1/L2 hit model ----
// KernelScope backend doc, simulator/engine.py: "Cache parameters" (128-byte
// lines; L1 1024 lines, hit 28 cycles; L2 49152 lines, hit 150 cycles; DRAM
// 400) and SimpleCache, a direct-mapped cache: the set of a line is
// line % num_lines, an access hits when the set's tag is that line, and a
// miss installs it. (The page's LRU list never picks a victim in a
// direct-mapped cache, so it is left out.) One L1 and one L2 serve the whole
// grid, as the page's simulator holds one of each.
struct SimpleCache {
  std::vector<int64_t> tags;  // per set: the cached line, -1 = empty
  explicit SimpleCache(uint32_t lines) : tags(lines, -1) {}
  bool access(uint64_t line) {
    int64_t& t = tags[(size_t)(line % tags.size())];
    if (t == (int64_t)line) return true;
    t = (int64_t)line;
    return false;
  }
};

struct CacheModel {
  SimpleCache l1, l2;
  uint32_t lat_l1, lat_l2;
  CacheModel(uint32_t n1, uint32_t n2, uint32_t a1, uint32_t a2) : l1(n1), l2(n2), lat_l1(a1), lat_l2(a2) {}
  // the page's _execute_instruction: L1 first, L2 on an L1 miss
  uint32_t access(uint64_t line) {
    if (l1.access(line)) return ORC_CACHE_L1_HIT;
    if (l2.access(line)) return ORC_CACHE_L2_HIT;
    return ORC_CACHE_DRAM;
  }
};

struct CacheAccess { uint64_t line; uint64_t step; uint32_t level; };

// ------------------------------------------------- shared memory (per CTA) ----

struct CtaMem {
  std::vector<uint8_t> bytes;  // zeroed at the start of the CTA
  // race checker state per 4-byte word, cleared at every barrier release
  bool race_on = false;
  std::vector<int64_t> writer, reader;
  uint32_t race_flags = 0;

  CtaMem(uint32_t size, bool race) : bytes(size, 0), race_on(race) {
    if (race_on) {
      writer.assign(size / 4 + 1, -1);
      reader.assign(size / 4 + 1, -1);
    }
  }
  void new_interval() {
    if (!race_on) return;
    std::fill(writer.begin(), writer.end(), -1);
    std::fill(reader.begin(), reader.end(), -1);
  }
  void note(uint64_t off, uint32_t size, int64_t gtid, bool write) {
    if (!race_on) return;
    for (uint64_t w = off / 4; w < (off + size + 3) / 4; w++) {
      int64_t& wr = writer[(size_t)w];
      int64_t& rd = reader[(size_t)w];
      if (write) {
        if (wr >= 0 && wr != gtid) race_flags |= ORC_RACE_CROSS_THREAD;
        if (rd != -1 && rd != gtid) race_flags |= ORC_RACE_CROSS_THREAD;
        wr = gtid;
      } else {
        if (wr >= 0 && wr != gtid) race_flags |= ORC_RACE_CROSS_THREAD;
        if (rd == -1) rd = gtid; else if (rd != gtid) rd = -2;
      }
    }
  }
};

// The shared address of a lane: register (zero-extended) plus offset.
uint64_t shared_addr(const Inst& in, const Lane& L) {
  uint64_t base = in.a.reg >= 0 ? L.v[(size_t)in.a.reg] : 0;
  return base + (uint64_t)in.a.off;
}

// 0, or the status of a shared access of `size` bytes at `addr`.
int shared_check(uint64_t addr, uint32_t size, uint32_t shared_bytes) {
  if (addr % size != 0) return ORC_ST_MISALIGNED;
  if (shared_bytes < size || addr > (uint64_t)shared_bytes - size) return ORC_ST_OOB;
  return 0;
}

// Bank-conflict degree of one request over the executing lanes (the page's
// analyze_shared_memory_access, written out): lanes grouped by bank; a bank
// whose lanes all use one address is a broadcast and counts 1, any other bank
// counts its lanes; the request's degree is the largest count, at least 1.
uint32_t bank_degree(const uint64_t* addr, uint32_t exec) {
  std::map<uint64_t, std::vector<uint64_t>> banks;
  for (int i = 0; i < 32; i++)
    if ((exec >> i) & 1) banks[(addr[i] / 4) % 32].push_back(addr[i]);
  uint32_t worst = 1;
  for (const auto& kv : banks) {
    const std::vector<uint64_t>& a = kv.second;
    const bool broadcast = std::set<uint64_t>(a.begin(), a.end()).size() == 1;
    if (!broadcast) worst = std::max(worst, (uint32_t)a.size());
  }
  return worst;
}

// ---------------------------------------------------------- warp mode ----

struct Entry { int pc, rpc; uint32_t mask; };

// What WarpRun::run stopped on.
enum { RUN_DONE = 0, RUN_BAR = 1, RUN_STEP = 2, RUN_PEEK = 3 };

// What a warp's next instruction waits for, by the kind of result that
// arrives last (SM issue model): a load's, a div/sqrt's, or any other
// (including a branch's latency); loads count first, then div/sqrt.
enum { WAIT_EXEC = 0, WAIT_MATH = 1, WAIT_MEM = 2 };

// One simulated warp, resumable at barriers (and, for the cache model, after
// every instruction).
struct WarpRun {
  const Launch* X;
  uint32_t gwarp, cta, wic;
  std::vector<Lane> lanes;
  std::vector<LaneCtx> ctx;
  std::vector<Entry> stack;
  std::vector<uint64_t> ready;
  uint64_t t_next = 0, t_last = 0, max_ready = 0, drain = 0;
  orc_warp_stats st;
  uint32_t n_events = 0, n_dropped = 0;
  std::vector<std::pair<uint32_t, uint64_t>> records;  // (id << 24 | ts, payload)
  uint64_t step = 0;                  // cache model: the step of the next instruction
  std::vector<CacheAccess> accesses;  // cache model: this warp's accesses in order
  uint64_t floor = 0;                 // SM issue model: the cycle its scheduler issues it at
  std::vector<int> rkind;             // SM issue model: WAIT_* kind of each register's producer
  uint64_t peek_e = 0;                // SM issue model: scoreboard time of the next instruction
  int peek_kind = WAIT_EXEC;          //                 and what binds it
  bool labels = false;                // SM issue model: count the divergence label
  uint64_t diverged = 0;              // instructions issued while some live lane waited on the stack

  WarpRun(const Launch& L, uint32_t gw) : X(&L), gwarp(gw) {
    const Kernel& K = *X->K;
    cta = gwarp / X->warps_per_cta;
    wic = gwarp % X->warps_per_cta;
    lanes.resize(32);
    ctx.resize(32);
    uint32_t mask0 = 0;
    for (uint32_t i = 0; i < 32; i++) {
      lanes[i].v.assign(K.regs.size(), 0);
      ctx[i] = LaneCtx{wic * 32 + i, X->block, cta, X->grid, i};
      if (wic * 32 + i < X->block) mask0 |= 1u << i;
    }
    stack.push_back(Entry{0, (int)K.code.size(), mask0});
    ready.assign(K.regs.size(), 0);
    rkind.assign(K.regs.size(), WAIT_EXEC);
    std::memset(&st, 0, sizeof st);
    st.max_stack_depth = 1;
  }

  // Interprets until the warp finishes (RUN_DONE) or issues bar.sync (RUN_BAR,
  // with the issue cycle in *arrival). With one_step it also stops before a
  // second instruction would issue (RUN_STEP); a call that issues the
  // warp's last instruction returns RUN_DONE, so a warp is done in the step of
  // its last instruction.
  int run(Memory& M, CtaMem* S, uint64_t* arrival, bool one_step = false, bool peek = false) {
    const Kernel& K = *X->K;
    const orc_config& cfg = *X->cfg;
    const int n = (int)K.code.size();
    bool issued = false;
    while (!stack.empty()) {
      Entry& top = stack.back();
      if (top.pc == top.rpc || top.mask == 0) { stack.pop_back(); continue; }
      if (top.pc >= n) { top.mask = 0; continue; }  // virtual exit: remaining lanes finish
      const int pc = top.pc;
      const Inst& in = K.code[(size_t)pc];

      if (in.k == K_EVENT) {  // zero-cost pseudo-op
        if (n_events != 0xFFFFFFFFu) n_events++;
        if (records.size() < cfg.max_ts_per_warp) {
          uint64_t payload = 0;  // the lowest active lane's register
          if (in.a.k == Opnd::REG)
            for (int i = 0; i < 32; i++)
              if ((top.mask >> i) & 1) { payload = lanes[(size_t)i].v[(size_t)in.a.reg]; break; }
          records.push_back({((uint32_t)(in.event & 0xFF) << 24) | (uint32_t)(t_next & 0xFFFFFF), payload});
        }
        else if (n_dropped < 0xFFFF)
          n_dropped++;
        top.pc = pc + 1;
        continue;
      }
      if (one_step && issued) return RUN_STEP;
      if (cfg.inject_warp >= 0 && (uint64_t)cfg.inject_warp == gwarp && st.warp_insts == cfg.inject_step) {
        st.status = ORC_ST_INJECTED;
        return RUN_DONE;
      }
      if (st.warp_insts == cfg.step_limit) { st.status = ORC_ST_STEP_LIMIT; return RUN_DONE; }
      if (peek) {  // the next instruction's scoreboard time, without issuing it
        std::vector<int> regs;
        auto use = [&](const Opnd& o) { if ((o.k == Opnd::REG || o.k == Opnd::MEM) && o.reg >= 0) regs.push_back(o.reg); };
        if (in.k == K_STG || in.k == K_STS) { use(in.a); use(in.b); }
        else if (in.k != K_BRA && in.k != K_RET && in.k != K_BAR) {
          use(in.a); use(in.b); use(in.c);
          regs.push_back(in.d.reg);
        }
        if (in.guard >= 0) regs.push_back(in.guard);
        uint64_t e = t_next;
        for (int r : regs) e = std::max(e, ready[(size_t)r]);
        int kind = WAIT_EXEC;
        for (int r : regs) if (ready[(size_t)r] == e) kind = std::max(kind, rkind[(size_t)r]);
        peek_e = e;
        peek_kind = kind;
        return RUN_PEEK;
      }
      issued = true;
      if (labels) {  // DIVERGENCE: live lanes (in any stack entry) outside the active mask
        uint32_t live = 0;
        for (const Entry& e : stack) live |= e.mask;
        if (live != top.mask) diverged++;
      }

      // ---- guard ----
      uint32_t exec = 0;
      for (int i = 0; i < 32; i++) {
        if (!((top.mask >> i) & 1)) continue;
        bool g = true;
        if (in.guard >= 0) g = (lanes[(size_t)i].v[(size_t)in.guard] != 0) != in.guard_neg;
        if (g) exec |= 1u << i;
      }
      uint64_t lat = cfg.lat[in.cls];

      // ---- cache model: one access at the lowest executing lane's line ----
      if (X->cache && (in.k == K_LDG || in.k == K_STG) && exec != 0) {
        int rep = 0;
        while (!((exec >> rep) & 1)) rep++;
        const uint64_t addr = lanes[(size_t)rep].v[(size_t)in.a.reg] + (uint64_t)in.a.off;
        const uint64_t line = addr / 128;
        const uint32_t level = X->cache->access(line);
        accesses.push_back(CacheAccess{line, step, level});
        if (in.k == K_LDG)
          lat = level == ORC_CACHE_L1_HIT ? X->cache->lat_l1 : level == ORC_CACHE_L2_HIT ? X->cache->lat_l2 : lat;
      }

      // ---- issue: in-order scoreboard ----
      std::vector<int> srcs, dsts;
      auto src = [&](const Opnd& o) { if ((o.k == Opnd::REG || o.k == Opnd::MEM) && o.reg >= 0) srcs.push_back(o.reg); };
      if (in.k == K_STG || in.k == K_STS) { src(in.a); src(in.b); }
      else if (in.k != K_BRA && in.k != K_RET && in.k != K_BAR) {
        src(in.a); src(in.b); src(in.c);
        dsts.push_back(in.d.reg);
      }
      if (in.guard >= 0) srcs.push_back(in.guard);
      uint64_t t = t_next;
      for (int r : srcs) t = std::max(t, ready[(size_t)r]);
      for (int r : dsts) t = std::max(t, ready[(size_t)r]);
      t = std::max(t, floor);
      const int produced = (in.k == K_LDG || in.k == K_LDS) ? WAIT_MEM : in.cls == ORC_LAT_SFU ? WAIT_MATH : WAIT_EXEC;
      for (int r : dsts) {
        ready[(size_t)r] = t + lat;
        rkind[(size_t)r] = produced;
        max_ready = std::max(max_ready, t + lat);
      }
      if (in.k == K_STG || in.k == K_STS) drain = std::max(drain, t + lat);
      t_last = t;
      t_next = (in.k == K_BRA || in.k == K_RET) ? t + lat : t + 1;
      st.warp_insts++;
      st.thread_insts += (uint64_t)popcount32(top.mask);

      // ---- execute ----
      if (in.k == K_BAR) {  // stop here until the CTA's barrier releases
        top.pc = pc + 1;
        *arrival = t;
        return RUN_BAR;
      }
      if (in.k == K_BRA) {
        uint32_t taken = exec, fall = top.mask & ~exec;
        if (fall == 0) { top.pc = in.target; }
        else if (taken == 0) { top.pc = pc + 1; }
        else {
          if (X->events)
            X->events->push_back(HintEvent{(uint32_t)pc, EV_DIVERGE, (uint32_t)popcount32(taken),
                                           (uint32_t)popcount32(fall), 0, 0});
          int R = K.ipdom[(size_t)pc];
          if (top.rpc == R) stack.pop_back(); else top.pc = R;
          bool overflow = false;
          if (in.target != R) {
            if (stack.size() >= cfg.stack_depth) overflow = true;
            else stack.push_back(Entry{in.target, R, taken});
          }
          if (!overflow && pc + 1 != R) {
            if (stack.size() >= cfg.stack_depth) overflow = true;
            else stack.push_back(Entry{pc + 1, R, fall});
          }
          if (overflow) { st.status = ORC_ST_SIMT_STACK; return RUN_DONE; }
          st.max_stack_depth = std::max(st.max_stack_depth, (uint32_t)stack.size());
        }
        continue;
      }
      if (in.k == K_RET) {
        for (Entry& e : stack) e.mask &= ~exec;
        stack.back().pc = pc + 1;
        continue;
      }
      if (in.k == K_LDG || in.k == K_STG) {
        uint32_t size = (uint32_t)width_of(in.ty) / 8;
        uint64_t addr[32];
        uint8_t* host[32];
        int bi[32];
        uint64_t off[32];
        int err = 0;
        for (int i = 0; i < 32 && !err; i++) {
          if (!((exec >> i) & 1)) continue;
          addr[i] = lanes[(size_t)i].v[(size_t)in.a.reg] + (uint64_t)in.a.off;
          err = M.translate(addr[i], size, &host[i], &bi[i], &off[i]);
        }
        if (err) { st.status = err; return RUN_DONE; }
        if (exec) {
          std::set<uint64_t> sectors, lines;
          for (int i = 0; i < 32; i++) {
            if (!((exec >> i) & 1)) continue;
            sectors.insert(addr[i] >> 5);
            lines.insert(addr[i] >> 7);
          }
          if (in.k == K_LDG) { st.ld_req++; st.ld_sectors += sectors.size(); st.ld_lines += lines.size(); }
          else { st.st_req++; st.st_sectors += sectors.size(); st.st_lines += lines.size(); }
          if (X->events)
            X->events->push_back(HintEvent{(uint32_t)pc, EV_GLOBAL, (uint32_t)popcount32(exec),
                                           (uint32_t)lines.size(), size, 0});
        }
        for (int i = 0; i < 32; i++) {  // ascending lanes: the highest lane's store lands last
          if (!((exec >> i) & 1)) continue;
          int64_t gtid = (int64_t)cta * X->block + ctx[(size_t)i].tid;
          if (in.k == K_LDG) {
            M.note(bi[i], off[i], size, gtid, false);
            lanes[(size_t)i].v[(size_t)in.d.reg] = load_le(host[i], size);
          } else {
            M.note(bi[i], off[i], size, gtid, true);
            store_le(host[i], lanes[(size_t)i].v[(size_t)in.b.reg], size);
          }
        }
        top.pc = pc + 1;
        continue;
      }
      if (in.k == K_LDS || in.k == K_STS) {
        uint32_t size = (uint32_t)width_of(in.ty) / 8;
        uint64_t addr[32];
        int err = 0;
        for (int i = 0; i < 32 && !err; i++) {
          if (!((exec >> i) & 1)) continue;
          addr[i] = shared_addr(in, lanes[(size_t)i]);
          err = shared_check(addr[i], size, K.shared_bytes);
        }
        if (err) { st.status = err; return RUN_DONE; }
        if (exec) {
          const uint32_t degree = bank_degree(addr, exec);
          st.sh_req++;
          st.sh_wavefronts += degree;
          if (X->events) X->events->push_back(HintEvent{(uint32_t)pc, EV_SHARED, degree, 0, 0, 0});
        }
        for (int i = 0; i < 32; i++) {  // ascending lanes: the highest lane's store lands last
          if (!((exec >> i) & 1)) continue;
          int64_t gtid = (int64_t)cta * X->block + ctx[(size_t)i].tid;
          uint8_t* p = S->bytes.data() + addr[i];
          if (in.k == K_LDS) {
            S->note(addr[i], size, gtid, false);
            lanes[(size_t)i].v[(size_t)in.d.reg] = load_le(p, size);
          } else {
            S->note(addr[i], size, gtid, true);
            store_le(p, lanes[(size_t)i].v[(size_t)in.b.reg], size);
          }
        }
        top.pc = pc + 1;
        continue;
      }
      for (int i = 0; i < 32; i++)
        if ((exec >> i) & 1) alu(in, lanes[(size_t)i], ctx[(size_t)i], X->params);
      top.pc = pc + 1;
    }
    return RUN_DONE;
  }

  void write_back() const {
    orc_warp_stats out = st;
    out.cycles = st.warp_insts ? std::max(std::max(t_last + 1, max_ready), drain) : 0;
    std::memcpy(X->stats + (uint64_t)gwarp * sizeof(orc_warp_stats), &out, sizeof out);
    if (X->trace) {
      uint8_t* slot = X->trace + (uint64_t)gwarp * X->slot_bytes;
      std::memset(slot, 0, X->slot_bytes);
      store_le(slot + 0, n_events, 4);
      const uint32_t rb = X->K->record_bytes;
      slot[4] = 1;
      slot[5] = (uint8_t)rb;
      store_le(slot + 6, n_dropped, 2);
      store_le(slot + 8, out.cycles, 8);
      // record layouts: [word] / [word | u32 payload] / [word | 0 | u64 payload]
      for (size_t i = 0; i < records.size(); i++) {
        uint8_t* r = slot + 16 + rb * i;
        store_le(r, records[i].first, 4);
        if (rb == 8) store_le(r + 4, records[i].second, 4);
        if (rb == 16) store_le(r + 8, records[i].second, 8);
      }
    }
    if (X->cache && X->cache_warps) {
      uint32_t l1 = 0, l2 = 0;
      for (const CacheAccess& a : accesses) {
        l1 += a.level == ORC_CACHE_L1_HIT;
        l2 += a.level == ORC_CACHE_L2_HIT;
      }
      const uint32_t n = (uint32_t)accesses.size();
      uint8_t* c = X->cache_warps + (uint64_t)gwarp * 16;
      store_le(c + 0, n, 4);
      store_le(c + 4, l1, 4);
      store_le(c + 8, l2, 4);
      store_le(c + 12, n - l1 - l2, 4);
      for (uint32_t k = 0; X->cache_log && k < n && k < X->cache_cap; k++) {
        uint8_t* r = X->cache_log + ((uint64_t)gwarp * X->cache_cap + k) * 16;
        store_le(r + 0, accesses[k].line, 8);
        store_le(r + 8, accesses[k].step, 4);
        store_le(r + 12, accesses[k].level, 4);
      }
    }
  }
};

// A warp of a kernel with no shared memory and no barrier runs alone.
void run_warp(const Launch& X, Memory& M, uint32_t gwarp) {
  WarpRun w(X, gwarp);
  uint64_t arrival;
  w.run(M, nullptr, &arrival);
  w.write_back();
}

// Every warp of one CTA, barrier interval by barrier interval (the page's
// step(): warps waiting at the barrier are skipped until all have arrived).
void run_cta(const Launch& X, Memory& M, uint32_t cta) {
  const Kernel& K = *X.K;
  CtaMem S(K.shared_bytes, M.race_on);
  std::vector<WarpRun> ws;
  for (uint32_t w = 0; w < X.warps_per_cta; w++) ws.emplace_back(X, cta * X.warps_per_cta + w);
  std::vector<char> done(ws.size(), 0), waiting(ws.size(), 0);
  for (;;) {
    bool any_waiting = false;
    uint64_t latest = 0;
    for (size_t w = 0; w < ws.size(); w++) {
      if (done[w]) continue;
      uint64_t arrival = 0;
      if (ws[w].run(M, &S, &arrival) == RUN_BAR) {
        waiting[w] = 1;
        any_waiting = true;
        latest = std::max(latest, arrival);
      } else {
        done[w] = 1;
      }
    }
    if (!any_waiting) break;  // every warp has finished
    const uint64_t release = latest + X.cfg->lat[ORC_LAT_BAR];
    for (size_t w = 0; w < ws.size(); w++)
      if (waiting[w]) { ws[w].t_next = release; waiting[w] = 0; }
    S.new_interval();
  }
  for (const WarpRun& w : ws) w.write_back();
  M.race_flags |= S.race_flags;
}

// ------------------------------------------------ stepper (cache model) ----
// The page's step()/run() taken literally: in every step each warp of the
// grid that is neither done nor waiting at a barrier executes one
// instruction, blocks in order and warps in order within a block; so global
// accesses reach the caches in (step, block, warp) order. A CTA whose warps
// are all waiting or done at the end of a step releases its barrier: the
// waiting warps resume (t_next = latest bar.sync issue + lat[bar]) and issue
// again in the next step. A warp is done in the step of its last
// instruction.
void run_stepped(const Launch& X, Memory& M) {
  const Kernel& K = *X.K;
  const uint32_t W = X.grid * X.warps_per_cta;
  std::vector<WarpRun> ws;
  ws.reserve(W);
  for (uint32_t w = 0; w < W; w++) ws.emplace_back(X, w);
  std::vector<CtaMem> shared;
  if (K.cta_mode()) for (uint32_t c = 0; c < X.grid; c++) shared.emplace_back(K.shared_bytes, M.race_on);
  enum { RUNNING, WAITING, DONE };
  std::vector<int> state(W, RUNNING);
  std::vector<uint64_t> arrival(W, 0);
  uint32_t n_done = 0;
  for (uint64_t step = 0; n_done < W; step++) {
    for (uint32_t w = 0; w < W; w++) {
      if (state[w] != RUNNING) continue;
      ws[w].step = step;
      CtaMem* S = K.cta_mode() ? &shared[w / X.warps_per_cta] : nullptr;
      const int r = ws[w].run(M, S, &arrival[w], true);
      if (r == RUN_BAR) state[w] = WAITING;
      else if (r == RUN_DONE) { state[w] = DONE; n_done++; }
    }
    for (uint32_t c = 0; c < X.grid && K.cta_mode(); c++) {
      const uint32_t w0 = c * X.warps_per_cta, w1 = w0 + X.warps_per_cta;
      bool running = false, waiting = false;
      uint64_t latest = 0;
      for (uint32_t w = w0; w < w1; w++) {
        running |= state[w] == RUNNING;
        if (state[w] == WAITING) { waiting = true; latest = std::max(latest, arrival[w]); }
      }
      if (running || !waiting) continue;
      for (uint32_t w = w0; w < w1; w++)
        if (state[w] == WAITING) { ws[w].t_next = latest + X.cfg->lat[ORC_LAT_BAR]; state[w] = RUNNING; }
      shared[c].new_interval();
    }
  }
  for (const WarpRun& w : ws) w.write_back();
  for (const CtaMem& S : shared) M.race_flags |= S.race_flags;
}

// ------------------------------------------------- SM issue model ----
// Each SM cycle by cycle: CTA c runs on SM c % n_sm, ctas_per_sm of them at
// once, the next one starting in a slot when the slot's CTA has finished (the
// latest end of its warps); warp slot i issues on scheduler i % schedulers;
// every cycle each scheduler issues one instruction of its ready warp with
// the lowest global warp id, if any (the page's step() order). A warp is ready
// when its in-order scoreboard lets it issue (peek); it then issues at this
// cycle (floor). Waits are counted by what the warp waited for.
//
// Two labels on issued instructions (they change no timing): MEMORY_THROTTLE,
// an instruction of the page's memory class (its MEMORY_OPS: ld, st, mov)
// issued while at least 4 other warps of its SM have a memory operation
// pending — a warp's pending operation is its latest global or shared load
// or store, issued at an earlier cycle and not yet complete (a load's result
// not yet ready, a store not yet drained); and DIVERGENCE, an instruction
// issued while some of the warp's live lanes wait on the reconvergence stack.
struct SchedWarp {
  std::unique_ptr<WarpRun> w;
  int state = 0;  // 0 empty, 1 running, 2 waiting, 3 done
  uint64_t start = 0, end = 0, base = 0, arrival = 0;
  uint64_t not_selected = 0, stall[3] = {0, 0, 0}, stall_bar = 0;
  bool has_mem = false;                  // a global/shared access issued so far
  uint64_t mem_issue = 0, mem_done = 0;  // the latest one's issue cycle and completion
  bool has_prev = false;                 // the one before it (a warp issues once a cycle, so
  uint64_t prev_done = 0;                // the latest access before a cycle is one of the two)
  uint64_t throttled = 0;
  bool pending_at(uint64_t cycle) const {  // its latest access issued before `cycle` is incomplete
    if (!has_mem) return false;
    if (mem_issue < cycle) return mem_done > cycle;
    return has_prev && prev_done > cycle;
  }
};

bool page_memory_class(const Inst& in) {  // the page's MEMORY_OPS within the subset
  return in.k == K_LDP || in.k == K_LDG || in.k == K_LDS || in.k == K_STG || in.k == K_STS || in.k == K_MOV;
}

void run_sm_model(const Launch& X, Memory& M, uint32_t n_sm, uint32_t ctas_per_sm, uint32_t schedulers,
                  uint8_t* warps_out, uint8_t* sms_out) {
  const Kernel& K = *X.K;
  const uint32_t wpc = X.warps_per_cta;
  enum { EMPTY, RUNNING, WAITING, DONE };
  for (uint32_t sm = 0; sm < n_sm; sm++) {
    std::vector<SchedWarp> slot(ctas_per_sm * wpc);
    std::vector<std::unique_ptr<CtaMem>> smem(ctas_per_sm);
    uint32_t next_k = 0;
    uint64_t sm_end = 0, sm_issued = 0, ctas = 0;
    auto finish = [&](SchedWarp& q) {
      q.state = DONE;
      q.end = q.w->st.warp_insts ? std::max(std::max(q.w->t_last + 1, q.w->max_ready), q.w->drain) : q.start;
      uint8_t* r = warps_out + (uint64_t)q.w->gwarp * 80;
      const uint64_t v[10] = {q.start, q.end, q.w->st.warp_insts, q.not_selected, q.stall[WAIT_EXEC],
                              q.stall[WAIT_MEM], q.stall[WAIT_MATH], q.stall_bar, q.throttled, q.w->diverged};
      for (int i = 0; i < 10; i++) store_le(r + 8 * i, v[i], 8);
      q.w->write_back();  // statistics (cycles there are this model's absolute end)
      sm_end = std::max(sm_end, q.end);
      sm_issued += q.w->st.warp_insts;
    };
    auto peek = [&](SchedWarp& q) {  // no memory access before the issue
      uint64_t arr = 0;
      if (q.w->run(M, nullptr, &arr, true, true) == RUN_PEEK) q.state = RUNNING;
      else finish(q);
    };
    auto start_cta = [&](uint32_t c, uint64_t t0) {
      const uint64_t cta = sm + (uint64_t)(next_k++) * n_sm;
      for (uint32_t i = 0; i < wpc; i++) slot[c * wpc + i] = SchedWarp();
      if (cta >= X.grid) return;
      smem[c].reset(K.cta_mode() ? new CtaMem(K.shared_bytes, M.race_on) : nullptr);
      for (uint32_t i = 0; i < wpc; i++) {
        SchedWarp& q = slot[c * wpc + i];
        q.w.reset(new WarpRun(X, (uint32_t)cta * wpc + i));
        q.w->labels = true;
        q.w->t_next = t0;
        q.start = q.base = t0;
        q.state = RUNNING;
        peek(q);
      }
    };
    // release a barrier nobody runs towards; start the next CTA in a finished slot
    auto settle = [&](uint32_t c) {
      for (;;) {
        bool running = false, waiting = false, any = false;
        uint64_t latest = 0, fin = 0;
        for (uint32_t i = 0; i < wpc; i++) {
          const SchedWarp& q = slot[c * wpc + i];
          if (q.state == EMPTY) continue;
          any = true;
          running |= q.state == RUNNING;
          if (q.state == WAITING) { waiting = true; latest = std::max(latest, q.arrival); }
          if (q.state == DONE) fin = std::max(fin, q.end);
        }
        if (!any || running) return;
        if (waiting) {
          const uint64_t rel = latest + X.cfg->lat[ORC_LAT_BAR];
          for (uint32_t i = 0; i < wpc; i++) {
            SchedWarp& q = slot[c * wpc + i];
            if (q.state != WAITING) continue;
            q.stall_bar += rel - (q.arrival + 1);
            q.w->t_next = rel;
            q.base = rel;
            peek(q);
          }
          if (smem[c]) smem[c]->new_interval();
          continue;
        }
        if (smem[c]) M.race_flags |= smem[c]->race_flags;
        ctas++;
        start_cta(c, fin);
      }
    };
    for (uint32_t c = 0; c < ctas_per_sm; c++) {
      start_cta(c, 0);
      settle(c);
    }
    for (uint64_t cycle = 0;;) {
      bool live = false;
      for (uint32_t sch = 0; sch < schedulers; sch++) {
        SchedWarp* pick = nullptr;
        for (uint32_t i = sch; i < slot.size(); i += schedulers) {
          SchedWarp& q = slot[i];
          if (q.state == RUNNING || q.state == WAITING) live = true;
          if (q.state != RUNNING) continue;
          if (q.w->peek_e > cycle) continue;
          if (!pick || q.w->gwarp < pick->w->gwarp) pick = &q;
        }
        if (!pick) continue;
        SchedWarp& q = *pick;
        const uint32_t c = (uint32_t)((&q - slot.data()) / wpc);
        q.not_selected += cycle - q.w->peek_e;
        if (q.w->peek_e > q.base) q.stall[q.w->peek_kind] += q.w->peek_e - q.base;
        // the instruction about to issue (the peek stopped at it)
        const Inst& nx = K.code[(size_t)q.w->stack.back().pc];
        if (page_memory_class(nx)) {  // MEMORY_THROTTLE label
          uint32_t pending = 0;
          for (const SchedWarp& o : slot)
            if (&o != &q && o.state != EMPTY && o.pending_at(cycle)) pending++;
          if (pending >= 4) q.throttled++;
        }
        if (nx.k == K_LDG || nx.k == K_STG || nx.k == K_LDS || nx.k == K_STS) {  // issues at `cycle`
          q.has_prev = q.has_mem;
          q.prev_done = q.mem_done;
          q.has_mem = true;
          q.mem_issue = cycle;
          q.mem_done = cycle + X.cfg->lat[nx.cls];
        }
        q.w->floor = cycle;
        uint64_t arr = 0;
        const int r = q.w->run(M, smem[c].get(), &arr, true);
        q.base = cycle + 1;
        if (r == RUN_BAR) {
          q.state = WAITING;
          q.arrival = arr;
          settle(c);
        } else if (r == RUN_STEP) {
          peek(q);
          if (q.state == DONE) settle(c);
        } else {
          finish(q);
          settle(c);
        }
      }
      if (!live) break;
      // the next cycle at which some warp can issue
      uint64_t soonest = UINT64_MAX;
      for (const SchedWarp& q : slot)
        if (q.state == RUNNING) soonest = std::min(soonest, std::max(q.w->peek_e, cycle + 1));
      if (soonest == UINT64_MAX) {
        bool any = false;
        for (const SchedWarp& q : slot) any |= q.state == RUNNING || q.state == WAITING;
        if (!any) break;
        soonest = cycle + 1;
      }
      cycle = soonest;
    }
    const uint64_t v[3] = {sm_end, sm_issued, ctas};
    for (int i = 0; i < 3; i++) store_le(sms_out + (uint64_t)sm * 32 + 8 * i, v[i], 8);
    store_le(sms_out + (uint64_t)sm * 32 + 24, 0, 8);
  }
}

// ---------------------------------------------------- per-thread mode ----
// Each thread runs alone with scalar control flow (between barriers, in CTA
// kernels). Gives the memory image a race-free program must produce whatever
// the warp-level masking does.

struct ThreadRun {
  const Launch* X;
  uint32_t gwarp, lane, cta, wic;
  Lane L;
  LaneCtx c;
  int pc = 0;
  uint64_t steps = 0;
  int32_t status = 0;

  ThreadRun(const Launch& Xl, uint32_t gw, uint32_t ln) : X(&Xl), gwarp(gw), lane(ln) {
    cta = gwarp / X->warps_per_cta;
    wic = gwarp % X->warps_per_cta;
    L.v.assign(X->K->regs.size(), 0);
    c = LaneCtx{wic * 32 + lane, X->block, cta, X->grid, lane};
  }

  // Runs until the thread finishes (false) or reaches bar.sync (true).
  bool run(Memory& M, CtaMem* S) {
    const Kernel& K = *X->K;
    const int n = (int)K.code.size();
    while (pc < n) {
      const Inst& in = K.code[(size_t)pc];
      if (in.k == K_EVENT) { pc++; continue; }
      if (steps == X->cfg->step_limit) { status = ORC_ST_STEP_LIMIT; return false; }
      steps++;
      bool g = true;
      if (in.guard >= 0) g = (L.v[(size_t)in.guard] != 0) != in.guard_neg;
      if (in.k == K_BAR) { pc++; return true; }
      if (in.k == K_BRA) { pc = g ? in.target : pc + 1; continue; }
      if (in.k == K_RET) { if (g) return false; pc++; continue; }
      if (!g) { pc++; continue; }
      if (in.k == K_LDG || in.k == K_STG) {
        uint32_t size = (uint32_t)width_of(in.ty) / 8;
        uint64_t addr = L.v[(size_t)in.a.reg] + (uint64_t)in.a.off;
        uint8_t* host;
        int bi;
        uint64_t off;
        int err = M.translate(addr, size, &host, &bi, &off);
        if (err) { status = err; return false; }
        if (in.k == K_LDG) L.v[(size_t)in.d.reg] = load_le(host, size);
        else store_le(host, L.v[(size_t)in.b.reg], size);
        pc++;
        continue;
      }
      if (in.k == K_LDS || in.k == K_STS) {
        uint32_t size = (uint32_t)width_of(in.ty) / 8;
        uint64_t addr = shared_addr(in, L);
        int err = shared_check(addr, size, K.shared_bytes);
        if (err) { status = err; return false; }
        if (in.k == K_LDS) L.v[(size_t)in.d.reg] = load_le(S->bytes.data() + addr, size);
        else store_le(S->bytes.data() + addr, L.v[(size_t)in.b.reg], size);
        pc++;
        continue;
      }
      alu(in, L, c, X->params);
      pc++;
    }
    return false;
  }
};

// One warp's threads one after another (no shared memory, no barrier); or,
// in a CTA kernel, every thread of the CTA interval by interval. The status
// of each warp is that of its first failing thread in lane order.
void run_threads(const Launch& X, Memory& M, const std::vector<uint32_t>& warps, std::vector<int32_t>* status) {
  const Kernel& K = *X.K;
  CtaMem S(K.shared_bytes, false);
  if (!K.cta_mode()) {  // a failing thread stops its warp's remaining lanes
    for (size_t k = 0; k < warps.size(); k++) {
      const uint32_t wic = warps[k] % X.warps_per_cta;
      for (uint32_t lane = 0; lane < 32 && wic * 32 + lane < X.block; lane++) {
        ThreadRun t(X, warps[k], lane);
        t.run(M, &S);
        if (t.status) { (*status)[k] = t.status; break; }
      }
    }
    return;
  }
  std::vector<ThreadRun> ts;
  std::vector<size_t> owner;
  for (size_t k = 0; k < warps.size(); k++) {
    const uint32_t wic = warps[k] % X.warps_per_cta;
    for (uint32_t lane = 0; lane < 32 && wic * 32 + lane < X.block; lane++) {
      ts.emplace_back(X, warps[k], lane);
      owner.push_back(k);
    }
  }
  std::vector<char> done(ts.size(), 0);
  for (;;) {
    bool any_waiting = false;
    for (size_t i = 0; i < ts.size(); i++) {
      if (done[i]) continue;
      if (ts[i].run(M, &S)) any_waiting = true;
      else done[i] = 1;
    }
    if (!any_waiting) break;
  }
  for (size_t i = 0; i < ts.size(); i++) {
    int32_t& s = (*status)[owner[i]];
    if (!s && ts[i].status) s = ts[i].status;
  }
}

// ------------------------------------------------------------- driver ----

void copy_err(const std::string& m, char* err, uint64_t errlen) {
  if (!err || errlen == 0) return;
  size_t k = std::min<size_t>(m.size(), (size_t)errlen - 1);
  std::memcpy(err, m.data(), k);
  err[k] = 0;
}

}  // namespace

extern "C" {

void orc_config_default(orc_config* cfg) {
  std::memset(cfg, 0, sizeof *cfg);
  const uint32_t lat[ORC_NUM_LAT] = {4, 4, 400, 20, 8, 36, 1, 23, 23, 20, 0, 0};
  std::memcpy(cfg->lat, lat, sizeof lat);
  cfg->max_ts_per_warp = 0;
  cfg->stack_depth = 32;
  cfg->step_limit = 1ull << 26;
  cfg->inject_warp = -1;
  cfg->mode = ORC_MODE_WARP;
}

}  // extern "C"

namespace {

int run_impl(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
             const void* params, uint64_t param_bytes, const orc_buffer* bufs,
             uint32_t n_bufs, const orc_config* cfg, void* stats, void* trace,
             int32_t* status, uint32_t* race_flags, const orc_cache* cache, char* err, uint64_t errlen,
             std::vector<HintEvent>* events = nullptr) {
  try {
    if (!ptx || !kernel || !cfg || !stats || !status) throw OracleError{ORC_ERR_ARG, "null argument"};
    if (grid == 0 || block == 0 || block > 1024) throw OracleError{ORC_ERR_ARG, "bad launch shape"};
    if (n_bufs > 8) throw OracleError{ORC_ERR_ARG, "at most 8 buffers"};
    if (cfg->stack_depth == 0 || cfg->stack_depth > 32) throw OracleError{ORC_ERR_ARG, "stack depth must be 1..32"};
    for (uint32_t i = 0; i < n_bufs; i++) {
      if (bufs[i].sim_base % 4096 != 0 || bufs[i].bytes == 0 || !bufs[i].host)
        throw OracleError{ORC_ERR_ARG, "buffer base must be 4 KiB aligned and non-empty"};
      if (bufs[i].sim_base + bufs[i].bytes < bufs[i].sim_base) throw OracleError{ORC_ERR_ARG, "buffer wraps"};
      for (uint32_t j = 0; j < i; j++) {
        bool disjoint = bufs[i].sim_base + bufs[i].bytes <= bufs[j].sim_base ||
                        bufs[j].sim_base + bufs[j].bytes <= bufs[i].sim_base;
        if (!disjoint) throw OracleError{ORC_ERR_ARG, "buffers overlap"};
      }
    }
    Kernel K = load(std::string(ptx), std::string(kernel));
    if (param_bytes < K.param_bytes || (K.param_bytes && !params)) throw OracleError{ORC_ERR_ARG, "parameter block too small"};

    Launch X;
    X.K = &K;
    X.grid = grid;
    X.block = block;
    X.warps_per_cta = (block + 31) / 32;
    X.params = (const uint8_t*)params;
    X.cfg = cfg;
    X.stats = (uint8_t*)stats;
    X.trace = (uint8_t*)trace;
    X.slot_bytes = ((16ull + (uint64_t)K.record_bytes * cfg->max_ts_per_warp) + 7) / 8 * 8;
    const uint64_t W = (uint64_t)grid * X.warps_per_cta;
    std::unique_ptr<CacheModel> cm;
    if (cache) {
      if (cache->l1_lines == 0 || cache->l2_lines == 0) throw OracleError{ORC_ERR_ARG, "cache with no lines"};
      if (cfg->mode != ORC_MODE_WARP || cfg->n_warp_list)
        throw OracleError{ORC_ERR_ARG, "the cache model runs the whole grid in warp mode"};
      cm.reset(new CacheModel(cache->l1_lines, cache->l2_lines, cache->lat_l1, cache->lat_l2));
      X.cache = cm.get();
      X.cache_warps = (uint8_t*)cache->warps;
      X.cache_log = (uint8_t*)cache->log;
      X.cache_cap = cache->log_cap;
    }

    std::vector<uint32_t> warps;
    if (cfg->n_warp_list) {
      for (uint32_t i = 0; i < cfg->n_warp_list; i++) {
        if (cfg->warp_list[i] >= W) throw OracleError{ORC_ERR_ARG, "warp id outside the grid"};
        warps.push_back(cfg->warp_list[i]);
      }
    } else {
      for (uint64_t w = 0; w < W; w++) warps.push_back((uint32_t)w);
    }
    // Kernels with shared memory or barriers run whole CTAs: every warp of a
    // listed warp's CTA runs (and is written).
    const bool by_cta = K.cta_mode();
    std::vector<uint32_t> units;  // warps, or CTAs
    if (by_cta) {
      std::set<uint32_t> ctas;
      for (uint32_t w : warps) ctas.insert(w / X.warps_per_cta);
      units.assign(ctas.begin(), ctas.end());
      warps.clear();
      for (uint32_t c : units)
        for (uint32_t w = 0; w < X.warps_per_cta; w++) warps.push_back(c * X.warps_per_cta + w);
    } else {
      units = warps;
    }

    Memory M;
    M.bufs = bufs;
    M.n = n_bufs;
    if (cfg->race_check) {
      M.race_on = true;
      for (uint32_t i = 0; i < n_bufs; i++) {
        M.writer.emplace_back((size_t)(bufs[i].bytes / 4 + 1), -1);
        M.reader.emplace_back((size_t)(bufs[i].bytes / 4 + 1), -1);
      }
    }

    unsigned nthreads = cfg->threads ? cfg->threads : std::max(1u, std::thread::hardware_concurrency());
    if (cfg->race_check) nthreads = 1;
    X.events = events;
    if (events) nthreads = 1;
    nthreads = (unsigned)std::min<size_t>(nthreads, std::max<size_t>(1, units.size()));

    auto work = [&](size_t lo, size_t hi) {
      for (size_t k = lo; k < hi; k++) {
        if (cfg->mode == ORC_MODE_PER_THREAD) {
          std::vector<uint32_t> ws;
          if (by_cta) for (uint32_t w = 0; w < X.warps_per_cta; w++) ws.push_back(units[k] * X.warps_per_cta + w);
          else ws.push_back(units[k]);
          std::vector<int32_t> pst(ws.size(), 0);
          run_threads(X, M, ws, &pst);
          for (size_t j = 0; j < ws.size(); j++) {
            orc_warp_stats st;
            std::memset(&st, 0, sizeof st);
            st.status = pst[j];
            std::memcpy(X.stats + (uint64_t)ws[j] * sizeof st, &st, sizeof st);
          }
        } else if (by_cta) {
          run_cta(X, M, units[k]);
        } else {
          run_warp(X, M, units[k]);
        }
      }
    };
    if (cm) {
      run_stepped(X, M);
    } else if (nthreads <= 1) {
      work(0, units.size());
    } else {
      std::vector<std::thread> pool;
      size_t chunk = (units.size() + nthreads - 1) / nthreads;
      for (unsigned t = 0; t < nthreads; t++) {
        size_t lo = t * chunk, hi = std::min(units.size(), lo + chunk);
        if (lo < hi) pool.emplace_back(work, lo, hi);
      }
      for (std::thread& th : pool) th.join();
    }

    *status = 0;
    for (uint32_t w : warps) {
      int32_t s;
      std::memcpy(&s, X.stats + (uint64_t)w * sizeof(orc_warp_stats) + offsetof(orc_warp_stats, status), 4);
      if (s) { *status = s; break; }
    }
    if (race_flags) *race_flags = M.race_flags;
    copy_err("", err, errlen);
    return ORC_OK;
  } catch (const OracleError& e) {
    copy_err(e.msg, err, errlen);
    return e.code;
  } catch (const std::exception& e) {
    copy_err(e.what(), err, errlen);
    return ORC_ERR_ARG;
  }
}

}  // namespace

extern "C" {

int orc_run(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
            const void* params, uint64_t param_bytes, const orc_buffer* bufs,
            uint32_t n_bufs, const orc_config* cfg, void* stats, void* trace,
            int32_t* status, uint32_t* race_flags, char* err, uint64_t errlen) {
  return run_impl(ptx, kernel, grid, block, params, param_bytes, bufs, n_bufs, cfg, stats, trace, status,
                  race_flags, nullptr, err, errlen);
}

int orc_run_events(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
                   const void* params, uint64_t param_bytes, const orc_buffer* bufs,
                   uint32_t n_bufs, const orc_config* cfg, void* stats, void* trace,
                   int32_t* status, void* events, uint64_t events_cap, uint64_t* n_events,
                   char* err, uint64_t errlen) {
  if (!n_events) {
    copy_err("null n_events", err, errlen);
    return ORC_ERR_ARG;
  }
  std::vector<HintEvent> ev;
  const int rc = run_impl(ptx, kernel, grid, block, params, param_bytes, bufs, n_bufs, cfg, stats, trace, status,
                          nullptr, nullptr, err, errlen, &ev);
  *n_events = ev.size();
  if (rc == ORC_OK && events)
    std::memcpy(events, ev.data(), std::min<uint64_t>(ev.size(), events_cap) * sizeof(HintEvent));
  return rc;
}

int orc_run_sched(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
                  const void* params, uint64_t param_bytes, const orc_buffer* bufs,
                  uint32_t n_bufs, const orc_config* cfg, const orc_sched* sched, void* sched_warps,
                  void* sched_sms, void* stats_out, char* err, uint64_t errlen) {
  if (!sched || !sched_warps || !sched_sms) {
    copy_err("null argument", err, errlen);
    return ORC_ERR_ARG;
  }
  try {
    if (!ptx || !kernel || !cfg) throw OracleError{ORC_ERR_ARG, "null argument"};
    if (grid == 0 || block == 0 || block > 1024) throw OracleError{ORC_ERR_ARG, "bad launch shape"};
    const uint32_t wpc = (block + 31) / 32;
    const uint32_t ctas = sched->ctas_per_sm ? sched->ctas_per_sm : 32 / wpc;
    if (sched->n_sm == 0 || ctas == 0 || ctas * wpc > 32 ||
        !(sched->schedulers == 1 || sched->schedulers == 2 || sched->schedulers == 4))
      throw OracleError{ORC_ERR_ARG, "bad schedule configuration"};
    Kernel K = load(std::string(ptx), std::string(kernel));
    if (param_bytes < K.param_bytes || (K.param_bytes && !params)) throw OracleError{ORC_ERR_ARG, "parameter block too small"};
    Launch X;
    X.K = &K;
    X.grid = grid;
    X.block = block;
    X.warps_per_cta = wpc;
    X.params = (const uint8_t*)params;
    X.cfg = cfg;
    std::vector<uint8_t> stats((size_t)grid * wpc * sizeof(orc_warp_stats));
    X.stats = stats.data();
    X.trace = nullptr;
    X.slot_bytes = 0;
    Memory M;
    M.bufs = bufs;
    M.n = n_bufs;
    run_sm_model(X, M, sched->n_sm, ctas, sched->schedulers, (uint8_t*)sched_warps, (uint8_t*)sched_sms);
    if (stats_out) std::memcpy(stats_out, stats.data(), stats.size());
    copy_err("", err, errlen);
    return ORC_OK;
  } catch (const OracleError& e) {
    copy_err(e.msg, err, errlen);
    return e.code;
  }
}

int orc_run_cached(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
                   const void* params, uint64_t param_bytes, const orc_buffer* bufs,
                   uint32_t n_bufs, const orc_config* cfg, const orc_cache* cache, void* stats,
                   void* trace, int32_t* status, char* err, uint64_t errlen) {
  if (!cache) {
    copy_err("null cache", err, errlen);
    return ORC_ERR_ARG;
  }
  return run_impl(ptx, kernel, grid, block, params, param_bytes, bufs, n_bufs, cfg, stats, trace, status,
                  nullptr, cache, err, errlen);
}

int orc_ipdom(const char* ptx, const char* kernel, int32_t* out, uint32_t cap,
              uint32_t* n_out, char* err, uint64_t errlen) {
  try {
    Kernel K = load(std::string(ptx), std::string(kernel));
    *n_out = (uint32_t)K.code.size();
    for (size_t i = 0; i < K.ipdom.size() && i < cap; i++) out[i] = K.ipdom[i];
    return ORC_OK;
  } catch (const OracleError& e) {
    copy_err(e.msg, err, errlen);
    return e.code;
  }
}

int orc_params(const char* ptx, const char* kernel, uint32_t* offsets, uint32_t* sizes,
               uint32_t cap, uint32_t* n_params, uint32_t* param_bytes, char* err,
               uint64_t errlen) {
  try {
    Kernel K = load(std::string(ptx), std::string(kernel));
    *n_params = (uint32_t)K.params.size();
    *param_bytes = K.param_bytes;
    for (size_t i = 0; i < K.params.size() && i < cap; i++) {
      offsets[i] = K.params[i].off;
      sizes[i] = K.params[i].size;
    }
    return ORC_OK;
  } catch (const OracleError& e) {
    copy_err(e.msg, err, errlen);
    return e.code;
  }
}

int orc_event_info(const char* ptx, const char* kernel, uint32_t id, uint32_t* kind, uint32_t* payload_bytes,
                   char* name, uint64_t cap, char* err, uint64_t errlen) {
  try {
    Kernel K = load(std::string(ptx), std::string(kernel));
    if (id >= K.event_kind.size()) throw OracleError{ORC_ERR_NOT_FOUND, "no such event"};
    *kind = K.event_kind[id];
    *payload_bytes = K.event_payload[id];
    copy_err(K.event_name[id], name, cap);
    return ORC_OK;
  } catch (const OracleError& e) {
    copy_err(e.msg, err, errlen);
    return e.code;
  }
}

int orc_record_bytes(const char* ptx, const char* kernel, uint32_t* bytes, char* err, uint64_t errlen) {
  try {
    Kernel K = load(std::string(ptx), std::string(kernel));
    *bytes = K.record_bytes;
    return ORC_OK;
  } catch (const OracleError& e) {
    copy_err(e.msg, err, errlen);
    return e.code;
  }
}

int orc_events(const char* ptx, const char* kernel, uint32_t* kinds, uint32_t cap,
               uint32_t* n_events, char* err, uint64_t errlen) {
  try {
    Kernel K = load(std::string(ptx), std::string(kernel));
    *n_events = (uint32_t)K.event_kind.size();
    for (size_t i = 0; i < K.event_kind.size() && i < cap; i++) kinds[i] = K.event_kind[i];
    return ORC_OK;
  } catch (const OracleError& e) {
    copy_err(e.msg, err, errlen);
    return e.code;
  }
}

}  // extern "C"
