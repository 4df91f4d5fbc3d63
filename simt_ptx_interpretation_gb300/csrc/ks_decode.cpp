// ks_decode.cpp — host PTX-subset lexer, parser and decoder.
//
// Lowers the supported subset (KernelScope backend doc, "PTX Parser":
// directives, .entry/.param/.reg, instructions with an optional @%p / @!%p
// guard, opcode, modifier chain and operands) into the packed 32-byte KsInsn
// array the sm_103a interpreter executes, and computes each branch's
// reconvergence pc as its immediate post-dominator (Cooper, Harvey and
// Kennedy's iterative dominator algorithm run on the reversed CFG).
//
// Register allocation: a 32-bit register takes one 32-bit slot of the
// interpreter's shared-memory register file, a 64-bit register two
// consecutive slots; slots and predicate indices are assigned in order of
// first use. Immediates go to a per-kernel constant pool.
#include <algorithm>
#include <array>
#include <cctype>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "ks_internal.h"

namespace ks {
namespace {

struct Fail {
  int code;
  std::string msg;
};

[[noreturn]] void fail(int code, int line, const std::string& m) {
  throw Fail{code, "line " + std::to_string(line) + ": " + m};
}

// ------------------------------------------------------------------ lexer --

enum TokKind { TK_NAME, TK_NUM, TK_PUNCT, TK_PSEUDO, TK_EOF };

struct Tok {
  TokKind kind;
  std::string text;
  int line;
};

bool name_start(unsigned char c) { return std::isalpha(c) || c == '_' || c == '$' || c == '%' || c == '.'; }
bool name_char(unsigned char c) { return std::isalnum(c) || c == '_' || c == '$' || c == '.'; }

std::vector<Tok> lex(const char* p, size_t n) {
  std::vector<Tok> out;
  int line = 1;
  size_t i = 0;
  while (i < n) {
    unsigned char c = (unsigned char)p[i];
    if (c == '\n') { line++; i++; continue; }
    if (std::isspace(c)) { i++; continue; }
    if (c == '/' && i + 1 < n && p[i + 1] == '*') {
      size_t j = i + 2;
      while (j + 1 < n && !(p[j] == '*' && p[j + 1] == '/')) { if (p[j] == '\n') line++; j++; }
      if (j + 1 >= n) fail(KS_ERR_PARSE, line, "unterminated block comment");
      i = j + 2;
      continue;
    }
    if (c == '/' && i + 1 < n && p[i + 1] == '/') {
      size_t j = i + 2;
      while (j < n && p[j] != '\n') j++;
      std::string body(p + i + 2, j - i - 2);
      size_t a = 0;
      while (a < body.size() && std::isspace((unsigned char)body[a])) a++;
      if (body.compare(a, 5, "@iket") == 0) out.push_back({TK_PSEUDO, body.substr(a + 5), line});
      i = j;
      continue;
    }
    if (std::isdigit(c)) {
      size_t j = i;
      while (j < n && (std::isalnum((unsigned char)p[j]) || p[j] == '.' || p[j] == '_')) j++;
      out.push_back({TK_NUM, std::string(p + i, j - i), line});
      i = j;
      continue;
    }
    if (name_start(c)) {
      size_t j = i + 1;
      while (j < n && name_char((unsigned char)p[j])) j++;
      out.push_back({TK_NAME, std::string(p + i, j - i), line});
      i = j;
      continue;
    }
    if (std::strchr(",;:[](){}+-<>@!", (int)c)) {
      out.push_back({TK_PUNCT, std::string(1, (char)c), line});
      i++;
      continue;
    }
    fail(KS_ERR_PARSE, line, std::string("unexpected character '") + (char)c + "'");
  }
  out.push_back({TK_EOF, "", line});
  return out;
}

// ------------------------------------------------------------- literals ----

struct Lit {
  bool neg = false;
  uint64_t mag = 0;
  bool is_f32 = false;  // 0fXXXXXXXX
};

bool hexval(char ch, unsigned* v) {
  if (ch >= '0' && ch <= '9') { *v = (unsigned)(ch - '0'); return true; }
  if (ch >= 'a' && ch <= 'f') { *v = (unsigned)(ch - 'a' + 10); return true; }
  if (ch >= 'A' && ch <= 'F') { *v = (unsigned)(ch - 'A' + 10); return true; }
  return false;
}

bool parse_number(const std::string& s, Lit* out) {
  if (s.size() == 10 && s[0] == '0' && (s[1] == 'f' || s[1] == 'F')) {
    uint64_t v = 0;
    for (size_t i = 2; i < 10; i++) {
      unsigned d;
      if (!hexval(s[i], &d)) return false;
      v = (v << 4) | d;
    }
    out->mag = v;
    out->is_f32 = true;
    return true;
  }
  std::string t = s;
  if (!t.empty() && (t.back() == 'U' || t.back() == 'u')) t.pop_back();
  if (t.empty()) return false;
  uint64_t v = 0;
  if (t.size() > 2 && t[0] == '0' && (t[1] == 'x' || t[1] == 'X')) {
    if (t.size() > 18) return false;
    for (size_t i = 2; i < t.size(); i++) {
      unsigned d;
      if (!hexval(t[i], &d)) return false;
      v = (v << 4) | d;
    }
  } else {
    for (char ch : t) {
      if (ch < '0' || ch > '9') return false;
      uint64_t d = (uint64_t)(ch - '0');
      if (v > (~0ull - d) / 10) return false;
      v = v * 10 + d;
    }
  }
  out->mag = v;
  return true;
}

bool is_ident(const std::string& s) {
  if (s.empty()) return false;
  unsigned char c0 = (unsigned char)s[0];
  if (!(std::isalpha(c0) || c0 == '_' || c0 == '$')) return false;
  for (unsigned char c : s)
    if (!(std::isalnum(c) || c == '_' || c == '$')) return false;
  return true;
}

// --------------------------------------------------------------- types ----

enum PType { PT_BAD, PT_U32, PT_S32, PT_B32, PT_F32, PT_U64, PT_S64, PT_B64, PT_PRED };

PType ptype(const std::string& s) {
  static const std::map<std::string, PType> m = {
      {"u32", PT_U32}, {"s32", PT_S32}, {"b32", PT_B32}, {"f32", PT_F32},
      {"u64", PT_U64}, {"s64", PT_S64}, {"b64", PT_B64}, {"pred", PT_PRED}};
  auto it = m.find(s);
  return it == m.end() ? PT_BAD : it->second;
}
unsigned bits(PType t) {
  switch (t) {
    case PT_U32: case PT_S32: case PT_B32: case PT_F32: return 32;
    case PT_U64: case PT_S64: case PT_B64: return 64;
    case PT_PRED: return 1;
    default: return 0;
  }
}
bool integer(PType t) { return t == PT_U32 || t == PT_S32 || t == PT_U64 || t == PT_S64; }
bool is_signed(PType t) { return t == PT_S32 || t == PT_S64; }

// ------------------------------------------------------------ operands ----

struct Operand {
  enum Kind { NONE, REG, LIT, SPECIAL, MEM, PARAM, LABEL } kind = NONE;
  std::string name;  // register / label / param / base register
  Lit lit;           // LIT
  int special = 0;
  int64_t offset = 0;
};

struct RegDecl {
  unsigned width;   // 32, 64 or 1 (predicate)
  int index = -1;   // slot (first slot for 64-bit) or predicate index, -1 until used
};

// A statement of the kernel body after parsing.
struct Stmt {
  int line;
  bool pseudo = false;
  std::string pseudo_kind, pseudo_name, pseudo_payload;  // payload: a register, or empty
  std::string guard;  // predicate register name, empty if none
  bool guard_neg = false;
  std::string opcode;                 // base opcode
  std::vector<std::string> mods;      // modifiers after the base
  std::vector<Operand> ops;
};

struct KernelText {
  std::string name;
  int line;
  std::vector<std::pair<std::string, PType>> params;
  std::map<std::string, RegDecl> regs;
  std::vector<Stmt> body;
  std::map<std::string, size_t> labels;  // label -> index into body
  std::map<std::string, uint32_t> shared;  // .shared array -> shared address
  uint32_t shared_bytes = 0;
};

// --------------------------------------------------------------- parser ----

class Parser {
 public:
  explicit Parser(std::vector<Tok> t) : toks_(std::move(t)) {}

  std::vector<KernelText> module() {
    std::vector<KernelText> ks;
    while (cur().kind != TK_EOF) {
      const Tok& t = cur();
      if (t.kind != TK_NAME) fail(KS_ERR_UNSUPPORTED, t.line, "unsupported top-level token '" + t.text + "'");
      if (t.text == ".version" || t.text == ".target") {
        skip_line();
      } else if (t.text == ".loc" || t.text == ".file") {
        skip_line();
      } else if (t.text == ".address_size") {
        int ln = t.line;
        pos_++;
        if (cur().kind != TK_NUM || cur().text != "64") fail(KS_ERR_UNSUPPORTED, ln, "only .address_size 64 is supported");
        pos_++;
      } else if (t.text == ".visible") {
        pos_++;
      } else if (t.text == ".entry") {
        ks.push_back(entry());
      } else {
        fail(KS_ERR_UNSUPPORTED, t.line, "unsupported top-level statement " + t.text);
      }
    }
    return ks;
  }

 private:
  std::vector<Tok> toks_;
  size_t pos_ = 0;

  const Tok& cur() const { return toks_[pos_]; }
  const Tok& peek(size_t k = 1) const { return toks_[std::min(pos_ + k, toks_.size() - 1)]; }
  bool is(const char* punct) const { return cur().kind == TK_PUNCT && cur().text == punct; }
  void expect(const char* punct) {
    if (!is(punct)) fail(KS_ERR_PARSE, cur().line, std::string("expected '") + punct + "'");
    pos_++;
  }
  std::string name() {
    if (cur().kind != TK_NAME) fail(KS_ERR_PARSE, cur().line, "expected a name");
    return toks_[pos_++].text;
  }
  void skip_line() {
    int ln = cur().line;
    while (cur().kind != TK_EOF && cur().line == ln) pos_++;
  }

  KernelText entry() {
    KernelText k;
    k.line = cur().line;
    pos_++;  // .entry
    k.name = name();
    if (!is_ident(k.name)) fail(KS_ERR_PARSE, k.line, "bad kernel name");
    expect("(");
    std::set<std::string> seen;
    if (!is(")")) {
      while (true) {
        int ln = cur().line;
        if (cur().kind != TK_NAME || cur().text != ".param") fail(KS_ERR_UNSUPPORTED, ln, "unsupported parameter declaration");
        pos_++;
        std::string ty = name();
        PType t = ty.size() > 1 && ty[0] == '.' ? ptype(ty.substr(1)) : PT_BAD;
        if (t == PT_BAD || t == PT_PRED) fail(KS_ERR_UNSUPPORTED, ln, "unsupported parameter type " + ty);
        std::string pn = name();
        if (!is_ident(pn)) fail(KS_ERR_PARSE, ln, "bad parameter name");
        if (!seen.insert(pn).second) fail(KS_ERR_PARSE, ln, "parameter declared twice");
        k.params.push_back({pn, t});
        if (is(",")) { pos_++; continue; }
        if (!is(")")) fail(KS_ERR_UNSUPPORTED, ln, "unsupported parameter declaration");
        break;
      }
    }
    expect(")");
    while (cur().kind != TK_EOF && !is("{")) pos_++;  // performance directives are ignored
    expect("{");
    std::vector<std::string> pending;
    while (true) {
      const Tok& t = cur();
      if (t.kind == TK_EOF) fail(KS_ERR_PARSE, t.line, "missing '}'");
      if (t.kind == TK_PUNCT && t.text == "}") { pos_++; break; }
      if (t.kind == TK_PUNCT && t.text == "{") fail(KS_ERR_UNSUPPORTED, t.line, "nested blocks are not supported");
      if (t.kind == TK_PSEUDO) {
        Stmt s;
        s.line = t.line;
        s.pseudo = true;
        std::vector<std::string> w;
        std::string word;
        for (char ch : t.text + " ") {
          if (std::isspace((unsigned char)ch)) { if (!word.empty()) w.push_back(word); word.clear(); }
          else word += ch;
        }
        if (w.size() != 2 && w.size() != 3) fail(KS_ERR_PARSE, t.line, "bad //@iket pseudo-op");
        s.pseudo_kind = w[0];
        s.pseudo_name = w[1];
        if (w.size() == 3) s.pseudo_payload = w[2];
        attach(k, pending, std::move(s));
        pos_++;
        continue;
      }
      if (t.kind == TK_NAME && (t.text == ".loc" || t.text == ".file")) { skip_line(); continue; }
      if (t.kind == TK_NAME && t.text == ".reg") { reg_decl(k); continue; }
      if (t.kind == TK_NAME && t.text == ".shared") { shared_decl(k); continue; }
      if (t.kind == TK_NAME && t.text[0] == '.') fail(KS_ERR_UNSUPPORTED, t.line, "unsupported directive in kernel body: " + t.text);
      if (t.kind == TK_NAME && peek().kind == TK_PUNCT && peek().text == ":" && is_ident(t.text)) {
        if (k.labels.count(t.text) || std::count(pending.begin(), pending.end(), t.text))
          fail(KS_ERR_PARSE, t.line, "label defined twice: " + t.text);
        pending.push_back(t.text);
        pos_ += 2;
        continue;
      }
      attach(k, pending, instruction());
    }
    if (!pending.empty()) fail(KS_ERR_PARSE, k.line, "label at the end of the kernel: " + pending[0]);
    return k;
  }

  static void attach(KernelText& k, std::vector<std::string>& pending, Stmt s) {
    for (const std::string& l : pending) k.labels[l] = k.body.size();
    pending.clear();
    k.body.push_back(std::move(s));
  }

  void reg_decl(KernelText& k) {
    int ln = cur().line;
    pos_++;
    std::string ty = name();
    PType t = ty.size() > 1 && ty[0] == '.' ? ptype(ty.substr(1)) : PT_BAD;
    if (t == PT_BAD) fail(KS_ERR_UNSUPPORTED, ln, "unsupported register type " + ty);
    while (true) {
      std::string rn = name();
      if (rn.size() < 2 || rn[0] != '%' || !is_ident(rn.substr(1))) fail(KS_ERR_PARSE, ln, "bad register name " + rn);
      std::vector<std::string> names;
      if (is("<")) {
        pos_++;
        Lit n;
        if (cur().kind != TK_NUM || !parse_number(cur().text, &n) || n.is_f32 || n.mag == 0 || n.mag > 4096)
          fail(KS_ERR_PARSE, ln, "bad register count");
        pos_++;
        expect(">");
        for (uint64_t i = 0; i < n.mag; i++) names.push_back(rn + std::to_string(i));
      } else {
        names.push_back(rn);
      }
      for (const std::string& r : names) {
        if (k.regs.count(r)) fail(KS_ERR_PARSE, ln, "register declared twice: " + r);
        k.regs[r] = RegDecl{bits(t)};
      }
      if (is(",")) { pos_++; continue; }
      break;
    }
    expect(";");
  }

  // .shared [.align A] .TYPE name[[N]];  arrays laid out in declaration order
  // from shared address 0, each at its alignment (the type's size by default)
  void shared_decl(KernelText& k) {
    const int ln = cur().line;
    pos_++;
    uint64_t align = 0;
    if (cur().kind == TK_NAME && cur().text == ".align") {
      pos_++;
      Lit a;
      if (cur().kind != TK_NUM || !parse_number(cur().text, &a) || a.is_f32 || a.mag == 0 || (a.mag & (a.mag - 1)) ||
          a.mag > 4096)
        fail(KS_ERR_PARSE, ln, "bad .align");
      align = a.mag;
      pos_++;
    }
    const std::string ty = name();
    static const std::map<std::string, uint32_t> esz = {
        {".b8", 1}, {".u8", 1}, {".s8", 1}, {".b16", 2}, {".u16", 2}, {".s16", 2},
        {".b32", 4}, {".u32", 4}, {".s32", 4}, {".f32", 4},
        {".b64", 8}, {".u64", 8}, {".s64", 8}, {".f64", 8}};
    auto et = esz.find(ty);
    if (et == esz.end()) fail(KS_ERR_UNSUPPORTED, ln, "unsupported .shared type " + ty);
    const std::string nm = name();
    if (!is_ident(nm)) fail(KS_ERR_PARSE, ln, "bad .shared name");
    uint64_t count = 1;
    if (is("[")) {
      pos_++;
      Lit c;
      if (cur().kind != TK_NUM || !parse_number(cur().text, &c) || c.is_f32 || c.mag == 0 || c.mag > (1u << 20))
        fail(KS_ERR_PARSE, ln, "bad .shared array size");
      count = c.mag;
      pos_++;
      expect("]");
    }
    expect(";");
    if (k.shared.count(nm)) fail(KS_ERR_PARSE, ln, "shared array declared twice: " + nm);
    if (!align) align = et->second;
    const uint64_t off = (k.shared_bytes + align - 1) / align * align;
    const uint64_t end = off + count * et->second;
    if (end > KS_MAX_SHARED_BYTES) fail(KS_ERR_UNSUPPORTED, ln, "more than 48 KiB of shared memory");
    k.shared[nm] = (uint32_t)off;
    k.shared_bytes = (uint32_t)end;
  }

  Stmt instruction() {
    Stmt s;
    s.line = cur().line;
    if (is("@")) {
      pos_++;
      if (is("!")) { s.guard_neg = true; pos_++; }
      s.guard = name();
      if (s.guard[0] != '%') fail(KS_ERR_PARSE, s.line, "bad guard");
    }
    std::string op = name();
    if (op[0] == '%' || op[0] == '.') fail(KS_ERR_PARSE, s.line, "expected an opcode");
    size_t dot = op.find('.');
    s.opcode = op.substr(0, dot);
    while (dot != std::string::npos) {
      size_t nd = op.find('.', dot + 1);
      s.mods.push_back(op.substr(dot + 1, nd == std::string::npos ? std::string::npos : nd - dot - 1));
      dot = nd;
    }
    if (!is(";")) {
      while (true) {
        s.ops.push_back(operand());
        if (is(",")) { pos_++; continue; }
        break;
      }
    }
    expect(";");
    return s;
  }

  Operand operand() {
    Operand o;
    int ln = cur().line;
    if (is("[")) {
      pos_++;
      o.name = name();
      o.kind = o.name[0] == '%' ? Operand::MEM : Operand::PARAM;
      if (is("+") || is("-")) {
        int sign = is("-") ? -1 : 1;
        pos_++;
        if (is("-")) { sign = -sign; pos_++; }
        Lit l;
        if (cur().kind != TK_NUM || !parse_number(cur().text, &l) || l.is_f32 || l.mag > 0x7FFFFFFFull)
          fail(KS_ERR_PARSE, ln, "bad address offset");
        pos_++;
        o.offset = sign * (int64_t)l.mag;
      }
      expect("]");
      return o;
    }
    if (is("-")) {
      pos_++;
      if (cur().kind != TK_NUM || !parse_number(cur().text, &o.lit) || o.lit.is_f32) fail(KS_ERR_PARSE, ln, "bad literal");
      o.lit.neg = true;
      o.kind = Operand::LIT;
      pos_++;
      return o;
    }
    if (cur().kind == TK_NUM) {
      if (!parse_number(cur().text, &o.lit)) fail(KS_ERR_PARSE, ln, "bad literal " + cur().text);
      o.kind = Operand::LIT;
      pos_++;
      return o;
    }
    std::string n = name();
    if (n[0] == '%') {
      static const std::map<std::string, int> sp = {
          {"%tid.x", SP_TID}, {"%ntid.x", SP_NTID}, {"%ctaid.x", SP_CTAID}, {"%nctaid.x", SP_NCTAID},
          {"%laneid", SP_LANEID}, {"%tid.y", SP_ZERO}, {"%tid.z", SP_ZERO}, {"%ctaid.y", SP_ZERO},
          {"%ctaid.z", SP_ZERO}, {"%ntid.y", SP_ONE}, {"%ntid.z", SP_ONE}, {"%nctaid.y", SP_ONE},
          {"%nctaid.z", SP_ONE}};
      auto it = sp.find(n);
      if (it != sp.end()) { o.kind = Operand::SPECIAL; o.special = it->second; return o; }
      o.kind = Operand::REG;
      o.name = n;
      return o;
    }
    if (!is_ident(n)) fail(KS_ERR_PARSE, ln, "bad operand " + n);
    o.kind = Operand::LABEL;
    o.name = n;
    return o;
  }
};

// -------------------------------------------------------------- decoder ----

class Decoder {
 public:
  Decoder(KernelText& t, KsKernel& k) : T(t), K(k) {}

  void run() {
    K.name = T.name;
    uint32_t off = 0;
    for (auto& p : T.params) {
      uint32_t sz = bits(p.second) / 8;
      off = (off + sz - 1) / sz * sz;
      K.params.push_back({p.first, off, sz});
      off += sz;
    }
    K.param_bytes = off;
    K.shared_bytes = T.shared_bytes;
    if (T.body.empty()) fail(KS_ERR_PARSE, T.line, "empty kernel");
    if (T.body.size() > KS_MAX_INSNS) fail(KS_ERR_LIMIT, T.line, "kernel longer than 2048 entries");
    for (Stmt& s : T.body) K.code.push_back(s.pseudo ? event(s) : insn(s));
    // branch targets
    for (size_t i = 0; i < T.body.size(); i++) {
      const Stmt& s = T.body[i];
      if (s.pseudo || s.opcode != "bra") continue;
      auto it = T.labels.find(s.ops[0].name);
      if (it == T.labels.end()) fail(KS_ERR_PARSE, s.line, "undefined label " + s.ops[0].name);
      K.code[i].target = (uint32_t)it->second;
    }
    const KsInsn& last = K.code.back();
    if (!((last.op == OP_RET || last.op == OP_BRA) && last.guard == KS_NO_GUARD))
      fail(KS_ERR_PARSE, T.body.back().line, "control can fall off the end of the kernel");
    K.n_slots = next_slot_;
    K.n_preds = next_pred_;
    postdominators();
    for (size_t i = 0; i < K.code.size(); i++)
      if (K.code[i].op == OP_BRA) K.code[i].rpc = (uint32_t)K.ipdom[i];
    build_image();
  }

 private:
  KernelText& T;
  KsKernel& K;
  uint32_t next_slot_ = 0, next_pred_ = 0;
  std::map<uint64_t, uint32_t> consts_;
  std::map<std::pair<uint32_t, std::string>, uint32_t> event_ids_;

  KsInsn blank() {
    KsInsn in;
    std::memset(&in, 0, sizeof in);
    in.guard = KS_NO_GUARD;
    in.hd = in.ha = in.hb = in.hc = in.hg = KS_HZ_NONE;
    in.lat = KS_LAT_ALU;
    return in;
  }

  KsInsn event(const Stmt& s) {
    uint32_t kind;
    if (s.pseudo_kind == "mark") kind = 0;
    else if (s.pseudo_kind == "range_start") kind = 1;
    else if (s.pseudo_kind == "range_end") kind = 2;
    else fail(KS_ERR_PARSE, s.line, "unknown //@iket kind " + s.pseudo_kind);
    if (!is_ident(s.pseudo_name)) fail(KS_ERR_PARSE, s.line, "bad event name");
    // optional payload register (IKET payload events): its value in the
    // warp's lowest active lane goes into the record
    uint32_t pbytes = 0;
    uint8_t preg = 0;
    if (!s.pseudo_payload.empty()) {
      if (s.pseudo_payload[0] != '%') fail(KS_ERR_PARSE, s.line, "an //@iket payload must be a register");
      RegDecl& r = reg(s.pseudo_payload, s.line);
      if (r.width != 32 && r.width != 64) fail(KS_ERR_PARSE, s.line, "an //@iket payload must be a 32- or 64-bit register");
      pbytes = r.width / 8;
      preg = (uint8_t)r.index;
    }
    auto key = std::make_pair(kind, s.pseudo_name);
    auto it = event_ids_.find(key);
    uint32_t id;
    if (it == event_ids_.end()) {
      id = (uint32_t)K.events.size();
      if (id >= 256) fail(KS_ERR_UNSUPPORTED, s.line, "more than 256 events");
      event_ids_[key] = id;
      K.events.push_back({s.pseudo_name, kind, pbytes});
    } else {
      id = it->second;
      if (K.events[id].payload_bytes != pbytes)
        fail(KS_ERR_PARSE, s.line, "event " + s.pseudo_name + " used with two payload sizes");
    }
    // NativeDump record sizes: 4 without a payload, 4 + 4, or 16
    K.record_bytes = std::max(K.record_bytes, pbytes == 0 ? 4u : pbytes == 4 ? 8u : 16u);
    KsInsn in = blank();
    in.op = OP_EVENT;
    in.event = (uint16_t)id;
    in.a = preg;
    in.flags = (uint8_t)pbytes;
    return in;
  }

  RegDecl& reg(const std::string& n, int line) {
    auto it = T.regs.find(n);
    if (it == T.regs.end()) fail(KS_ERR_PARSE, line, "undeclared register " + n);
    RegDecl& r = it->second;
    if (r.index < 0) {
      if (r.width == 1) {
        if (next_pred_ >= KS_MAX_PREDS) fail(KS_ERR_LIMIT, line, "more than 31 predicate registers in use");
        r.index = (int)next_pred_++;
      } else {
        uint32_t need = r.width / 32;
        if (next_slot_ + need > KS_MAX_SLOTS) fail(KS_ERR_LIMIT, line, "more than 96 register slots in use");
        r.index = (int)next_slot_;
        next_slot_ += need;
      }
    }
    return r;
  }

  uint8_t constant(uint64_t v, int line) {
    auto it = consts_.find(v);
    if (it != consts_.end()) return (uint8_t)(KS_CONST_BIT | it->second);
    if (K.cpool.size() >= KS_MAX_CONSTS) fail(KS_ERR_LIMIT, line, "more than 128 distinct immediates");
    uint32_t i = (uint32_t)K.cpool.size();
    K.cpool.push_back(v);
    consts_[v] = i;
    return (uint8_t)(KS_CONST_BIT | i);
  }

  // Predicate operand: returns the predicate index, sets the hazard index.
  uint8_t pred(const Operand& o, int line, uint8_t* hz) {
    if (o.kind != Operand::REG) fail(KS_ERR_PARSE, line, "predicate register expected");
    RegDecl& r = reg(o.name, line);
    if (r.width != 1) fail(KS_ERR_PARSE, line, "predicate register expected");
    *hz = (uint8_t)(KS_HZ_PRED0 + r.index);
    return (uint8_t)r.index;
  }

  // Destination register of `width` bits.
  uint8_t dest(const Operand& o, unsigned width, int line, uint8_t* hz) {
    if (o.kind != Operand::REG) fail(KS_ERR_PARSE, line, "register operand expected");
    RegDecl& r = reg(o.name, line);
    if (r.width != width) fail(KS_ERR_PARSE, line, "register width does not match the instruction type");
    *hz = (uint8_t)r.index;
    return (uint8_t)r.index;
  }

  // Source operand. allow: 'r' register only, 'v' register or literal,
  // 'm' register, literal or special register (mov).
  uint8_t source(const Operand& o, unsigned width, PType ty, char allow, int line, uint8_t* hz, int* special) {
    *hz = KS_HZ_NONE;
    switch (o.kind) {
      case Operand::REG: {
        RegDecl& r = reg(o.name, line);
        if (r.width != width) fail(KS_ERR_PARSE, line, "register width does not match the instruction type");
        *hz = (uint8_t)r.index;
        return (uint8_t)r.index;
      }
      case Operand::SPECIAL:
        if (allow != 'm' || width != 32) fail(KS_ERR_PARSE, line, "special register only allowed as a 32-bit mov source");
        *special = o.special;
        return 0;
      case Operand::LIT: {
        if (allow == 'r') fail(KS_ERR_PARSE, line, "register operand expected");
        uint64_t v;
        if (o.lit.is_f32) {
          if (!(ty == PT_F32 || ty == PT_B32)) fail(KS_ERR_PARSE, line, "f32 literal on a non-32-bit-float operand");
          v = o.lit.mag;
        } else {
          if (ty == PT_F32) fail(KS_ERR_PARSE, line, "f32 operands take 0fXXXXXXXX literals only");
          if (width == 32) {
            if (o.lit.neg ? o.lit.mag > 0x80000000ull : o.lit.mag > 0xFFFFFFFFull)
              fail(KS_ERR_PARSE, line, "literal does not fit 32 bits");
            v = (o.lit.neg ? (0 - o.lit.mag) : o.lit.mag) & 0xFFFFFFFFull;
          } else {
            if (o.lit.neg && o.lit.mag > 0x8000000000000000ull) fail(KS_ERR_PARSE, line, "literal does not fit 64 bits");
            v = o.lit.neg ? (0 - o.lit.mag) : o.lit.mag;
          }
        }
        return constant(v, line);
      }
      default:
        fail(KS_ERR_PARSE, line, "bad operand kind");
    }
  }

  KsInsn insn(const Stmt& s) {
    KsInsn in = blank();
    const int ln = s.line;
    if (!s.guard.empty()) {
      RegDecl& g = reg(s.guard, ln);
      if (g.width != 1) fail(KS_ERR_PARSE, ln, "guard must be a predicate");
      in.guard = (uint8_t)g.index;
      in.gneg = s.guard_neg ? 1 : 0;
      in.hg = (uint8_t)(KS_HZ_PRED0 + g.index);
    }
    const std::string& op = s.opcode;
    const std::vector<std::string>& m = s.mods;
    const std::vector<Operand>& o = s.ops;
    auto unsupported = [&]() -> void {
      std::string full = op;
      for (const std::string& x : m) full += "." + x;
      fail(KS_ERR_UNSUPPORTED, ln, "unsupported instruction form: " + full);
    };
    auto arity = [&](size_t n) {
      if (o.size() != n) fail(KS_ERR_PARSE, ln, op + ": expected " + std::to_string(n) + " operands");
    };
    int sp = -1;

    if (op == "add" || op == "sub" || op == "mul" || op == "mad" || op == "fma" || op == "div" || op == "sqrt") {
      bool rn = false, lo = false;
      PType t = PT_BAD;
      for (const std::string& x : m) {
        if (x == "rn" && !rn) rn = true;
        else if (x == "lo" && !lo) lo = true;
        else if (t == PT_BAD && ptype(x) != PT_BAD) t = ptype(x);
        else unsupported();
      }
      if (t == PT_BAD) unsupported();
      bool f = (t == PT_F32);
      size_t nops = 3;
      if (op == "add" || op == "sub") {
        if (lo || (!f && (!integer(t) || rn))) unsupported();
        in.op = f ? (op == "add" ? OP_FADD : OP_FSUB)
                  : bits(t) == 32 ? (op == "add" ? OP_ADD32 : OP_SUB32) : (op == "add" ? OP_ADD64 : OP_SUB64);
      } else if (op == "mul") {
        if (f ? lo : (!integer(t) || !lo || rn)) unsupported();
        in.op = f ? OP_FMUL : bits(t) == 32 ? OP_MUL32 : OP_MUL64;
      } else if (op == "mad") {
        if (!integer(t) || !lo || rn) unsupported();
        in.op = bits(t) == 32 ? OP_MAD32 : OP_MAD64;
        nops = 4;
      } else if (op == "fma") {
        if (!f || !rn || lo) unsupported();
        in.op = OP_FFMA;
        in.lat = KS_LAT_FMA;
        nops = 4;
      } else if (op == "div") {
        if (!f || !rn || lo) unsupported();
        in.op = OP_FDIV;
        in.lat = KS_LAT_SFU;
      } else {
        if (!f || !rn || lo) unsupported();
        in.op = OP_FSQRT;
        in.lat = KS_LAT_SFU;
        nops = 2;
      }
      arity(nops);
      unsigned w = bits(t);
      in.d = dest(o[0], w, ln, &in.hd);
      in.a = source(o[1], w, t, 'v', ln, &in.ha, &sp);
      if (nops > 2) in.b = source(o[2], w, t, 'v', ln, &in.hb, &sp);
      if (nops > 3) in.c = source(o[3], w, t, 'v', ln, &in.hc, &sp);
      return in;
    }
    if (op == "and" || op == "or" || op == "xor") {
      if (m.size() != 1) unsupported();
      PType t = ptype(m[0]);
      if (!(t == PT_B32 || t == PT_B64 || t == PT_PRED)) unsupported();
      arity(3);
      int k = op == "and" ? 0 : op == "or" ? 1 : 2;
      if (t == PT_PRED) {
        in.op = (uint8_t)(OP_ANDP + k);
        uint8_t hz;
        in.d = pred(o[0], ln, &in.hd);
        in.a = pred(o[1], ln, &hz); in.ha = hz;
        in.b = pred(o[2], ln, &hz); in.hb = hz;
      } else {
        in.op = (uint8_t)((t == PT_B32 ? OP_AND32 : OP_AND64) + k);
        unsigned w = bits(t);
        in.d = dest(o[0], w, ln, &in.hd);
        in.a = source(o[1], w, t, 'v', ln, &in.ha, &sp);
        in.b = source(o[2], w, t, 'v', ln, &in.hb, &sp);
      }
      return in;
    }
    if (op == "shl" || op == "shr") {
      if (m.size() != 1) unsupported();
      PType t = ptype(m[0]);
      if (op == "shl") {
        if (!(t == PT_B32 || t == PT_B64)) unsupported();
        in.op = t == PT_B32 ? OP_SHL32 : OP_SHL64;
      } else {
        if (!(t == PT_B32 || t == PT_B64 || integer(t))) unsupported();
        bool w32 = bits(t) == 32;
        in.op = is_signed(t) ? (w32 ? OP_SHR32S : OP_SHR64S) : (w32 ? OP_SHR32U : OP_SHR64U);
      }
      arity(3);
      unsigned w = bits(t);
      in.d = dest(o[0], w, ln, &in.hd);
      in.a = source(o[1], w, t, 'v', ln, &in.ha, &sp);
      in.b = source(o[2], 32, PT_U32, 'v', ln, &in.hb, &sp);
      return in;
    }
    if (op == "cvt") {
      std::vector<std::string> mm = m;
      int rnd = -1;  // -1 none, 4 = rn, else RND_*
      if (!mm.empty()) {
        if (mm[0] == "rn") rnd = 4;
        else if (mm[0] == "rni") rnd = RND_RNI;
        else if (mm[0] == "rzi") rnd = RND_RZI;
        else if (mm[0] == "rmi") rnd = RND_RMI;
        else if (mm[0] == "rpi") rnd = RND_RPI;
        if (rnd >= 0) mm.erase(mm.begin());
      }
      if (mm.size() != 2) unsupported();
      PType dt = ptype(mm[0]), st = ptype(mm[1]);
      arity(2);
      if (integer(dt) && integer(st)) {
        if (rnd >= 0) unsupported();
        unsigned dw = bits(dt), sw = bits(st);
        in.d = dest(o[0], dw, ln, &in.hd);
        in.a = source(o[1], sw, st, 'r', ln, &in.ha, &sp);
        if (dw == sw) in.op = dw == 32 ? OP_MOV32 : OP_MOV64;
        else if (dw == 64) in.op = is_signed(st) ? OP_CVT_SX : OP_CVT_ZX;
        else in.op = OP_MOV32;  // 64 -> 32 keeps the low slot
        return in;
      }
      if (dt == PT_F32 && integer(st)) {
        if (rnd != 4) unsupported();
        in.op = st == PT_U32 ? OP_CVT_F32_U32 : st == PT_S32 ? OP_CVT_F32_S32 : st == PT_U64 ? OP_CVT_F32_U64 : OP_CVT_F32_S64;
        in.d = dest(o[0], 32, ln, &in.hd);
        in.a = source(o[1], bits(st), st, 'r', ln, &in.ha, &sp);
        return in;
      }
      if (integer(dt) && st == PT_F32) {
        if (rnd < 0 || rnd == 4) unsupported();
        in.op = OP_CVT_F2I;
        uint8_t dk = dt == PT_S32 ? CVT_S32 : dt == PT_U32 ? CVT_U32 : dt == PT_S64 ? CVT_S64 : CVT_U64;
        in.flags = (uint8_t)(dk | (rnd << 4));
        in.d = dest(o[0], bits(dt), ln, &in.hd);
        in.a = source(o[1], 32, st, 'r', ln, &in.ha, &sp);
        return in;
      }
      unsupported();
    }
    if (op == "mov") {
      if (m.size() != 1) unsupported();
      PType t = ptype(m[0]);
      if (t == PT_BAD || t == PT_PRED) unsupported();
      arity(2);
      unsigned w = bits(t);
      in.d = dest(o[0], w, ln, &in.hd);
      Operand src = o[1];
      if (src.kind == Operand::LABEL) {  // the shared address of an array
        auto it = T.shared.find(src.name);
        if (it == T.shared.end() || t == PT_F32) fail(KS_ERR_PARSE, ln, "bad mov operand " + src.name);
        src.kind = Operand::LIT;
        src.lit = Lit{};
        src.lit.mag = it->second;
      }
      in.a = source(src, w, t, 'm', ln, &in.ha, &sp);
      if (sp >= 0) {
        in.op = OP_MOVSP;
        in.imm = (uint64_t)sp;
      } else {
        in.op = w == 32 ? OP_MOV32 : OP_MOV64;
      }
      in.flags = KS_MOV_OPCODE;
      return in;
    }
    if (op == "setp") {
      if (m.size() != 2) unsupported();
      const std::string& c = m[0];
      PType t = ptype(m[1]);
      bool uname = (c == "lo" || c == "ls" || c == "hi" || c == "hs");
      uint8_t cmp;
      if (c == "eq") cmp = CMP_EQ;
      else if (c == "ne") cmp = CMP_NE;
      else if (c == "lt" || c == "lo") cmp = CMP_LT;
      else if (c == "le" || c == "ls") cmp = CMP_LE;
      else if (c == "gt" || c == "hi") cmp = CMP_GT;
      else if (c == "ge" || c == "hs") cmp = CMP_GE;
      else unsupported();
      if (t == PT_B32 || t == PT_B64) { if (!(cmp == CMP_EQ || cmp == CMP_NE)) unsupported(); }
      else if (t == PT_U32 || t == PT_U64) { }
      else if (t == PT_S32 || t == PT_S64 || t == PT_F32) { if (uname) unsupported(); }
      else unsupported();
      in.op = t == PT_F32 ? OP_SETP_F32
              : t == PT_S32 ? OP_SETP_S32
              : t == PT_S64 ? OP_SETP_S64
              : bits(t) == 32 ? OP_SETP_U32 : OP_SETP_U64;
      in.flags = cmp;
      arity(3);
      unsigned w = bits(t);
      in.d = pred(o[0], ln, &in.hd);
      in.a = source(o[1], w, t, 'v', ln, &in.ha, &sp);
      in.b = source(o[2], w, t, 'v', ln, &in.hb, &sp);
      return in;
    }
    if (op == "selp") {
      if (m.size() != 1) unsupported();
      PType t = ptype(m[0]);
      if (t == PT_BAD || t == PT_PRED) unsupported();
      arity(4);
      unsigned w = bits(t);
      in.op = w == 32 ? OP_SELP32 : OP_SELP64;
      in.d = dest(o[0], w, ln, &in.hd);
      in.a = source(o[1], w, t, 'v', ln, &in.ha, &sp);
      in.b = source(o[2], w, t, 'v', ln, &in.hb, &sp);
      in.c = pred(o[3], ln, &in.hc);
      return in;
    }
    if (op == "bra") {
      if (!(m.empty() || (m.size() == 1 && m[0] == "uni"))) unsupported();
      arity(1);
      if (o[0].kind != Operand::LABEL) fail(KS_ERR_PARSE, ln, "bra needs a label");
      in.op = OP_BRA;
      in.lat = KS_LAT_BRA;
      return in;
    }
    if (op == "ret" || op == "exit") {
      if (!m.empty()) unsupported();
      arity(0);
      in.op = OP_RET;
      in.lat = KS_LAT_RET;
      return in;
    }
    if (op == "ld" || op == "st") {
      if (m.size() != 2) unsupported();
      PType t = ptype(m[1]);
      if (t == PT_BAD || t == PT_PRED) unsupported();
      unsigned w = bits(t);
      arity(2);
      if (op == "ld" && m[0] == "global") {
        in.op = w == 32 ? OP_LDG32 : OP_LDG64;
        in.lat = KS_LAT_LDG;
        in.d = dest(o[0], w, ln, &in.hd);
        address(o[1], ln, &in);
        return in;
      }
      if (op == "ld" && m[0] == "param") {
        in.op = w == 32 ? OP_LDP32 : OP_LDP64;
        in.d = dest(o[0], w, ln, &in.hd);
        if (o[1].kind != Operand::PARAM) fail(KS_ERR_PARSE, ln, "ld.param needs [param(+offset)]");
        const KsParam* p = nullptr;
        for (const KsParam& q : K.params) if (q.name == o[1].name) p = &q;
        if (!p) fail(KS_ERR_PARSE, ln, "unknown parameter " + o[1].name);
        int64_t at = (int64_t)p->offset + o[1].offset;
        int64_t sz = w / 8;
        if (at < 0 || at + sz > (int64_t)K.param_bytes || at % sz) fail(KS_ERR_PARSE, ln, "ld.param outside the parameter block or misaligned");
        in.imm = (uint64_t)at;
        return in;
      }
      if (op == "st" && m[0] == "global") {
        in.op = w == 32 ? OP_STG32 : OP_STG64;
        in.lat = KS_LAT_STG;
        address(o[0], ln, &in);
        in.b = source(o[1], w, t, 'r', ln, &in.hb, &sp);
        return in;
      }
      if (op == "ld" && m[0] == "shared") {
        in.op = w == 32 ? OP_LDS32 : OP_LDS64;
        in.lat = KS_LAT_LDS;
        in.d = dest(o[0], w, ln, &in.hd);
        shared_address(o[1], ln, &in);
        return in;
      }
      if (op == "st" && m[0] == "shared") {
        in.op = w == 32 ? OP_STS32 : OP_STS64;
        in.lat = KS_LAT_STS;
        shared_address(o[0], ln, &in);
        in.b = source(o[1], w, t, 'r', ln, &in.hb, &sp);
        return in;
      }
      unsupported();
    }
    if (op == "bar" || op == "barrier") {
      // bar.sync 0 / barrier.sync[.aligned] 0: CTA barrier 0 over every thread
      const bool form = (op == "bar" && m.size() == 1 && m[0] == "sync") ||
                        (op == "barrier" && (m.size() == 1 || m.size() == 2) && m[0] == "sync" &&
                         (m.size() == 1 || m[1] == "aligned"));
      if (!form) unsupported();
      arity(1);
      if (o[0].kind != Operand::LIT || o[0].lit.neg || o[0].lit.is_f32 || o[0].lit.mag != 0)
        fail(KS_ERR_UNSUPPORTED, ln, "only barrier 0 without a thread count is supported");
      if (in.guard != KS_NO_GUARD) fail(KS_ERR_UNSUPPORTED, ln, "guarded bar.sync is not supported");
      in.op = OP_BAR;
      in.lat = KS_LAT_BAR;
      K.has_bar = true;
      return in;
    }
    fail(KS_ERR_UNSUPPORTED, ln, "unsupported opcode " + op);
  }

  // [%r(+off)] with a 32- or 64-bit register, or [array(+off)]
  void shared_address(const Operand& o, int ln, KsInsn* in) {
    if (o.kind == Operand::PARAM) {
      auto it = T.shared.find(o.name);
      if (it == T.shared.end()) fail(KS_ERR_PARSE, ln, "unknown shared array " + o.name);
      in->flags = 0;
      in->imm = (uint64_t)((int64_t)it->second + o.offset);
      return;
    }
    if (o.kind != Operand::MEM) fail(KS_ERR_PARSE, ln, "shared address must be [register(+offset)] or [array(+offset)]");
    RegDecl& r = reg(o.name, ln);
    if (r.width != 32 && r.width != 64)
      fail(KS_ERR_PARSE, ln, "shared address must be [register(+offset)] or [array(+offset)]");
    in->a = (uint8_t)r.index;
    in->ha = (uint8_t)r.index;
    in->flags = (uint8_t)(KS_SHA_REG | (r.width == 64 ? KS_SHA_WIDE : 0));
    in->imm = (uint64_t)o.offset;  // sign-extended
  }

  void address(const Operand& o, int ln, KsInsn* in) {
    if (o.kind != Operand::MEM) fail(KS_ERR_PARSE, ln, "global access needs [64-bit register(+offset)]");
    RegDecl& r = reg(o.name, ln);
    if (r.width != 64) fail(KS_ERR_PARSE, ln, "global access needs [64-bit register(+offset)]");
    in->a = (uint8_t)r.index;
    in->ha = (uint8_t)r.index;
    in->imm = (uint64_t)o.offset;  // sign-extended
  }

  // Immediate post-dominators by Cooper-Harvey-Kennedy on the reverse CFG,
  // rooted at the virtual exit. Entries that cannot reach the exit
  // reconverge at the exit.
  void postdominators() {
    const int n = (int)K.code.size();
    const int EXIT = n;
    std::vector<std::vector<int>> succ((size_t)n + 1), pred((size_t)n + 1);
    for (int i = 0; i < n; i++) {
      const KsInsn& in = K.code[(size_t)i];
      bool guarded = in.guard != KS_NO_GUARD;
      std::vector<int>& s = succ[(size_t)i];
      if (in.op == OP_BRA) {
        s.push_back((int)in.target);
        if (guarded && (int)in.target != i + 1) s.push_back(i + 1);
      } else if (in.op == OP_RET) {
        s.push_back(EXIT);
        if (guarded) s.push_back(i + 1);
      } else {
        s.push_back(i + 1);
      }
      for (int x : s) pred[(size_t)x].push_back(i);
    }
    // postorder of the reverse graph (edges exit -> predecessors), iterative DFS
    std::vector<int> order, po_num((size_t)n + 1, -1);
    std::vector<char> seen((size_t)n + 1, 0);
    std::vector<std::pair<int, size_t>> stack;
    stack.push_back({EXIT, 0});
    seen[(size_t)EXIT] = 1;
    while (!stack.empty()) {
      auto& top = stack.back();
      const std::vector<int>& nb = pred[(size_t)top.first];
      if (top.second < nb.size()) {
        int v = nb[top.second++];
        if (!seen[(size_t)v]) { seen[(size_t)v] = 1; stack.push_back({v, 0}); }
      } else {
        po_num[(size_t)top.first] = (int)order.size();
        order.push_back(top.first);
        stack.pop_back();
      }
    }
    std::vector<int> idom((size_t)n + 1, -1);
    idom[(size_t)EXIT] = EXIT;
    auto intersect = [&](int a, int b) {
      while (a != b) {
        while (po_num[(size_t)a] < po_num[(size_t)b]) a = idom[(size_t)a];
        while (po_num[(size_t)b] < po_num[(size_t)a]) b = idom[(size_t)b];
      }
      return a;
    };
    bool changed = true;
    while (changed) {
      changed = false;
      for (int k = (int)order.size() - 1; k >= 0; k--) {  // reverse postorder
        int v = order[(size_t)k];
        if (v == EXIT) continue;
        int nd = -1;
        for (int s : succ[(size_t)v]) {  // predecessors in the reverse graph
          if (idom[(size_t)s] < 0) continue;
          nd = nd < 0 ? s : intersect(s, nd);
        }
        if (nd >= 0 && idom[(size_t)v] != nd) { idom[(size_t)v] = nd; changed = true; }
      }
    }
    K.ipdom.assign((size_t)n, EXIT);
    for (int i = 0; i < n; i++)
      if (seen[(size_t)i] && idom[(size_t)i] >= 0) K.ipdom[(size_t)i] = idom[(size_t)i];
  }

  // Width in bits of the row operand at position `pos` (0 a, 1 b, 2 c, 3 d)
  // of a decoded op, or 0 if that position holds no register/constant row.
  static unsigned row_width(const KsInsn& in, int pos) {
    const unsigned op = in.op;
    auto w = [&](unsigned a, unsigned b, unsigned c, unsigned d) {
      const unsigned v[4] = {a, b, c, d};
      return v[pos];
    };
    switch (op) {
      case OP_LDP32: return w(0, 0, 0, 32);
      case OP_LDP64: return w(0, 0, 0, 64);
      case OP_LDG32: return w(64, 0, 0, 32);
      case OP_LDG64: return w(64, 0, 0, 64);
      case OP_STG32: return w(64, 32, 0, 0);
      case OP_STG64: return w(64, 64, 0, 0);
      case OP_MOV32: return w(32, 0, 0, 32);
      case OP_MOV64: return w(64, 0, 0, 64);
      case OP_MOVSP: return w(0, 0, 0, 32);
      case OP_ADD32: case OP_SUB32: case OP_MUL32: case OP_AND32: case OP_OR32: case OP_XOR32:
      case OP_SHL32: case OP_SHR32U: case OP_SHR32S: case OP_FADD: case OP_FSUB: case OP_FMUL:
      case OP_FDIV: case OP_SELP32:
        return w(32, 32, 0, 32);
      case OP_MAD32: case OP_FFMA: return w(32, 32, 32, 32);
      case OP_ADD64: case OP_SUB64: case OP_MUL64: case OP_AND64: case OP_OR64: case OP_XOR64:
      case OP_SELP64:
        return w(64, 64, 0, 64);
      case OP_MAD64: return w(64, 64, 64, 64);
      case OP_SHL64: case OP_SHR64U: case OP_SHR64S: return w(64, 32, 0, 64);
      case OP_FSQRT: case OP_CVT_F32_U32: case OP_CVT_F32_S32: return w(32, 0, 0, 32);
      case OP_CVT_F32_U64: case OP_CVT_F32_S64: return w(64, 0, 0, 32);
      case OP_CVT_F2I: return w(32, 0, 0, ((in.flags & 15) == CVT_S64 || (in.flags & 15) == CVT_U64) ? 64 : 32);
      case OP_CVT_ZX: case OP_CVT_SX: return w(32, 0, 0, 64);
      case OP_SETP_U32: case OP_SETP_S32: case OP_SETP_F32: return w(32, 32, 0, 0);
      case OP_SETP_U64: case OP_SETP_S64: return w(64, 64, 0, 0);
      case OP_LDS32: case OP_LDS64: case OP_STS32: case OP_STS64: {
        const unsigned aw = (in.flags & KS_SHA_REG) ? ((in.flags & KS_SHA_WIDE) ? 64u : 32u) : 0u;
        const unsigned dw = op == OP_LDS32 || op == OP_STS32 ? 32u : 64u;
        return op == OP_LDS32 || op == OP_LDS64 ? w(aw, 0, 0, dw) : w(aw, dw, 0, 0);
      }
      case OP_EVENT: return w(in.flags * 8u, 0, 0, 0);  // the payload register, if any
      default: return 0;  // control, predicate logic, bar.sync
    }
  }

  // Routing constants of the unified datapaths (added to the pool on demand).
  static bool fpu_family(uint8_t op) { return op == OP_FADD || op == OP_FSUB || op == OP_FMUL || op == OP_FFMA; }
  static bool imad_family(uint8_t op) {
    return op == OP_ADD32 || op == OP_SUB32 || op == OP_MUL32 || op == OP_MAD32 || op == OP_MOV32;
  }

  // ops whose second operand is read as b | aux (aux = an immediate b, or 0)
  static bool imm_b_op(uint8_t op) {
    return op == OP_AND32 || op == OP_OR32 || op == OP_XOR32 || op == OP_SHL32 || op == OP_SHR32U ||
           op == OP_SHR32S || op == OP_SHL64 || op == OP_SHR64U || op == OP_SHR64S;
  }

  static unsigned routed_width(const KsInsn& in, int pos) {
    if (fpu_family(in.op) || imad_family(in.op)) return 32;
    return row_width(in, pos);
  }

  int in_line(size_t) const { return T.line; }

  // Lays out the warp region and emits the device image.
  // Operand routing of one instruction onto the unified datapaths (a, b, c
  // rows and the aux immediate).
  struct Route { uint8_t a, b, c; uint32_t aux; };

  // The program image of one layout (split = 0 PAIR, 1 SPLIT): the region
  // layout, one DevInsn per program entry plus the exit sentinel, the fast
  // runs' lengths and forwarding flags, and the constant row values.
  void resolve_image(uint32_t split, const std::vector<Route>& route, const std::vector<uint8_t>& madi,
                     const std::vector<uint32_t>& madi_c, const std::vector<uint32_t>& crow,
                     const std::vector<uint32_t>& rowval) {
    const size_t n = K.code.size();
    DevLayout& Y = K.layout[split];
    const uint32_t RB = split ? ROW_SPLIT : ROW_PAIR;
    Y.split = split;
    Y.row_bytes = RB;
    Y.n_slots = K.n_slots;
    Y.n_crows = (uint32_t)rowval.size();
    Y.const_off = K.n_slots * RB;
    Y.zero_off = Y.const_off + Y.n_crows * RB;
    const uint32_t n_rows = K.n_slots + Y.n_crows + 1u;
    if (split) {
      Y.ready_off = Y.zero_off + RB;
      Y.pred_off = Y.ready_off + n_rows * 4u;
      Y.n_ready = n_rows + 32u;
      Y.stack_off = (Y.pred_off + 32u * 4u + 7u) / 8u * 8u;
      Y.region_bytes = (Y.stack_off + KS_MAX_STACK * 8u + 127u) / 128u * 128u;
      // hazard offsets are 16-bit
      if (Y.region_bytes > 0xFFFFu) fail(KS_ERR_UNSUPPORTED, 0, "warp state beyond 64 KiB");
    } else {
      Y.ready_off = 0;
      Y.n_ready = 0;
      Y.pred_off = Y.zero_off + RB;
      Y.stack_off = Y.pred_off + 256u;
      Y.region_bytes = Y.stack_off + KS_MAX_STACK * 8u;
    }

    auto row_of = [&](uint8_t o) -> uint32_t {
      if (o == OPND_ZERO) return Y.zero_off;
      return (o & KS_CONST_BIT) ? Y.const_off + crow[o & 0x7F] * RB : (uint32_t)o * RB;
    };
    // predicate-table entry of a scoreboard index (the always-true
    // predicate's entry, which stays 0, when absent or not a predicate)
    auto phz = [&](uint8_t h) -> uint32_t {
      if (h != KS_HZ_NONE && h >= KS_HZ_PRED0) return Y.pred_entry(h - KS_HZ_PRED0);
      return Y.pred_entry(31);
    };
    auto pack = [](uint32_t lo, uint32_t hi) { return lo | (hi << 16); };
    // where the guard, its negation and DOP_MADII's immediate go
    uint32_t* (*guard_of)(DevInsn&) = split ? +[](DevInsn& o) { return &o.x[4]; } : +[](DevInsn& o) { return &o.x[0]; };
    uint32_t* (*gneg_of)(DevInsn&) = split ? +[](DevInsn& o) { return &o.x[5]; } : +[](DevInsn& o) { return &o.x[1]; };
    std::vector<DevInsn> dev(n + 1);
    for (size_t i = 0; i <= n; i++) {
      DevInsn& o = dev[i];
      std::memset(&o, 0, sizeof o);
      *guard_of(o) = 31;
      o.a = o.b = o.c = o.d = Y.zero_off;
      if (split) {
        const uint32_t z = Y.ready_of(Y.zero_off), p31 = Y.pred_entry(31);
        o.x[0] = o.x[1] = pack(z, z);
        o.x[2] = o.x[3] = pack(p31, p31);
      } else {
        o.x[2] = o.x[3] = o.x[4] = o.x[5] = Y.pred_entry(31);  // ha, hb, hc, hd
      }
      if (i == n) {  // exit sentinel
        o.op = OP_EXIT;
        continue;
      }
      const KsInsn& in = K.code[i];
      o.op = madi[i] ? (madi[i] == 1 ? DOP_MADI : DOP_MADII)
             : fpu_family(in.op) ? DOP_FPU : imad_family(in.op) ? DOP_IMAD : in.op;
      if ((o.op == DOP_FPU || o.op == DOP_IMAD) && in.guard != KS_NO_GUARD) o.op |= DOP_GUARDED;
      o.inc = in.op == OP_EVENT ? 0u : INC_ISSUE;
      if (in.guard != KS_NO_GUARD) {
        *guard_of(o) = in.guard;
        *gneg_of(o) = in.gneg ? 0xFFFFFFFFu : 0u;
      }
      const uint8_t ops[4] = {route[i].a, route[i].b, route[i].c, in.d};
      uint32_t* rows[4] = {&o.a, &o.b, &o.c, &o.d};
      for (int p = 0; p < 4; p++)
        if (routed_width(in, p)) *rows[p] = row_of(ops[p]);
      if ((o.op & ~DOP_GUARDED) == DOP_FPU || (o.op & ~DOP_GUARDED) == DOP_IMAD || imm_b_op(in.op) || madi[i])
        o.aux = route[i].aux;
      if (in.op != OP_EVENT) {
        const bool pdest = in.hd != KS_HZ_NONE && in.hd >= KS_HZ_PRED0;
        if (pdest) o.inc |= INC_PDEST;
        if (split) {
          // scoreboard terms: the rows read and written, the guard, the
          // predicate sources (the destination term is the predicate of
          // setp / predicate logic, which have no register destination)
          o.x[0] = pack(Y.ready_of(o.a), Y.ready_of(o.b));
          o.x[1] = pack(Y.ready_of(o.c), pdest ? phz(in.hd) : Y.ready_of(o.d));
          o.x[2] = pack(Y.pred_entry(*guard_of(o)), phz(in.ha));
          o.x[3] = pack(phz(in.hb), phz(in.hc));
        } else {
          // predicate hazards live in the predicate table; register hazards
          // travel with the register rows themselves
          o.x[2] = phz(in.ha);
          o.x[3] = phz(in.hb);
          o.x[4] = phz(in.hc);
          if (pdest) o.x[5] = phz(in.hd);
        }
        if (routed_width(in, 3)) o.inc |= INC_RDEST;
        const bool pred_operand = (in.ha >= KS_HZ_PRED0 && in.ha != KS_HZ_NONE) ||
                                  (in.hb >= KS_HZ_PRED0 && in.hb != KS_HZ_NONE) ||
                                  (in.hc >= KS_HZ_PRED0 && in.hc != KS_HZ_NONE) || pdest;
        if (pred_operand) o.inc |= INC_PHAZ;
        if (madi[i]) {
          o.inc |= INC_MID;  // unguarded, no predicate operand
          // DOP_MADII's immediate addend: x[4] in both layouts (PAIR: the
          // unused hc; SPLIT: the guard, whose term is already in hz)
          if (madi[i] == 2) o.x[4] = madi_c[i];
        }
        switch (in.op) {
          case OP_LDP32: case OP_LDP64: case OP_MOV64: case OP_MOVSP:
          case OP_ADD64: case OP_SUB64: case OP_MUL64: case OP_MAD64:
          case OP_AND32: case OP_OR32: case OP_XOR32: case OP_AND64: case OP_OR64: case OP_XOR64:
          case OP_SHL32: case OP_SHR32U: case OP_SHR32S: case OP_SHL64: case OP_SHR64U: case OP_SHR64S:
          case OP_FDIV: case OP_FSQRT:
          case OP_CVT_F32_U32: case OP_CVT_F32_S32: case OP_CVT_F32_U64: case OP_CVT_F32_S64:
          case OP_CVT_F2I: case OP_CVT_ZX: case OP_CVT_SX:
            if (in.guard == KS_NO_GUARD && !pred_operand) o.inc |= INC_MID;
            break;
          default:
            break;
        }
        switch (in.op) {  // the SM issue model's memory-throttle label
          case OP_LDG32: case OP_LDG64: case OP_STG32: case OP_STG64:
          case OP_LDS32: case OP_LDS64: case OP_STS32: case OP_STS64:
            o.inc |= INC_MCLASS | INC_MEMOP;
            break;
          case OP_LDP32: case OP_LDP64:
            o.inc |= INC_MCLASS;
            break;
          case OP_MOV32: case OP_MOV64: case OP_MOVSP:
            if (in.flags & KS_MOV_OPCODE) o.inc |= INC_MCLASS;
            break;
          default:
            break;
        }
        o.wlat = (uint32_t)in.lat;
        if (in.hd != KS_HZ_NONE) o.wlat |= DEV_HAS_DEST;
        if (in.op == OP_STG32 || in.op == OP_STG64 || in.op == OP_STS32 || in.op == OP_STS64) o.wlat |= DEV_IS_STORE;
        if (in.op == OP_BRA || in.op == OP_RET) o.wlat |= DEV_IS_CTRL;
      }
      switch (in.op) {
        case OP_EVENT: o.aux = in.event | ((uint32_t)in.flags << 8); break;
        case OP_LDG32: case OP_LDG64: case OP_STG32: case OP_STG64:
        case OP_LDP32: case OP_LDP64: case OP_MOVSP:
          o.aux = (uint32_t)in.imm;
          break;
        case OP_LDS32: case OP_LDS64: case OP_STS32: case OP_STS64:
          o.aux = (uint32_t)in.imm;
          if (in.flags & KS_SHA_WIDE) o.inc |= INC_ADDR64;
          break;
        case OP_CVT_F2I: o.aux = in.flags; break;
        case OP_SETP_U32: case OP_SETP_S32: case OP_SETP_U64: case OP_SETP_S64: case OP_SETP_F32: {
          o.aux = (uint32_t)in.flags | ((uint32_t)in.d << 8);
          const KsInsn* nx = i + 1 < n ? &K.code[i + 1] : nullptr;
          if (in.guard == KS_NO_GUARD && nx && nx->op == OP_BRA && nx->guard == in.d && nx->target < (1u << 15)) {
            o.inc |= INC_FUSE;
            o.aux |= ((uint32_t)(nx->gneg ? 1u : 0u) << 16) | (nx->target << 17);
          }
          break;
        }
        case OP_ANDP: case OP_ORP: case OP_XORP:
          o.aux = (uint32_t)in.a | ((uint32_t)in.b << 8) | ((uint32_t)in.d << 16);
          break;
        case OP_SELP32: case OP_SELP64: o.aux = in.c; break;
        case OP_BRA: o.aux = (in.target & 0xFFFFu) | ((in.rpc & 0xFFFFu) << 16); break;
        default: break;
      }
    }
    // run lengths of the fast path (unguarded routed FPU / IMAD ops)
    auto fast = [&](size_t i) { return dev[i].op == DOP_FPU || dev[i].op == DOP_IMAD; };
    for (size_t i = n; i-- > 0;) {
      DevInsn& o = dev[i];
      if (fast(i)) {
        const uint32_t next = fast(i + 1) ? (dev[i + 1].inc >> INC_RUN_SHIFT) : 0u;
        o.inc |= (next + 1u) << INC_RUN_SHIFT;
      }
    }
    // Short fast runs (at most MID_FAST_RUN ops, e.g. one address mad or a
    // hash step's mul and add between logic ops) run in the mid loop instead:
    // between mid ops they would cut its run in three, each piece taking a
    // dispatch, while the fast loop's pipelining only pays on long runs.
    for (size_t i = 0; i < n; i++) {
      if (!fast(i) || (i > 0 && fast(i - 1))) continue;  // the first op of a run
      const uint32_t len = dev[i].inc >> INC_RUN_SHIFT;
      if (len > MID_FAST_RUN) continue;
      for (size_t j = i; j < i + len; j++) dev[j].inc = (dev[j].inc & ((1u << INC_RUN_SHIFT) - 1u)) | INC_MID;
    }
    // forwarding flags between consecutive fast ops (read by the SPLIT fast
    // loop): inside a run the next op's operands and scoreboard terms are
    // loaded before this op's stores
    for (size_t i = 1; i < n; i++) {
      if (!fast(i) || !fast(i - 1)) continue;
      DevInsn& o = dev[i];
      const uint32_t pd = dev[i - 1].d;
      if (o.a == pd) o.inc |= INC_FWD_A;
      if (o.b == pd) o.inc |= INC_FWD_B;
      if (o.c == pd) o.inc |= INC_FWD_C;
      if (o.a == pd || o.b == pd || o.c == pd || o.d == pd) o.inc |= INC_FWD_T;
    }
    // runs (from each op to the run's end) whose ops all write a row they read
    for (size_t i = n; i-- > 0;) {
      DevInsn& o = dev[i];
      if ((o.inc >> INC_RUN_SHIFT) == 0u) continue;  // not in a fast run
      const bool own = o.d == o.a || o.d == o.b || o.d == o.c;
      const bool rest = (o.inc >> INC_RUN_SHIFT) == 1u || (dev[i + 1].inc & INC_OWN_D) != 0u;
      if (own && rest) o.inc |= INC_OWN_D;
    }
    // PAIR: how many ops from each run op on keep reading its b and c rows
    // (rows the op before does not write), and whether all of them are f32
    // ops, in x[4] (hc: fast ops have no predicate operands)
    if (!split) {
      for (size_t i = n; i-- > 0;) {
        DevInsn& o = dev[i];
        const uint32_t len = o.inc >> INC_RUN_SHIFT;
        if (len == 0u) continue;
        uint32_t keep = 1u;
        bool fpu = o.op == DOP_FPU;
        if (len > 1u) {
          const DevInsn& x = dev[i + 1];
          if (x.b == o.b && x.c == o.c && o.b != o.d && o.c != o.d) {
            keep = 1u + (x.x[4] & KEEP_COUNT);
            fpu = fpu && (x.x[4] & KEEP_FPU) != 0u;
          }
        }
        o.x[4] = keep | (fpu ? KEEP_FPU : 0u);
      }
    }
    K.prog_bytes = (uint32_t)((n + 1) * sizeof(DevInsn));
    const size_t cb = rowval.size() * 4;
    std::vector<uint8_t>& img = K.image[split];
    img.assign((K.prog_bytes + cb + 15) / 16 * 16, 0);
    std::memcpy(img.data(), dev.data(), K.prog_bytes);
    if (cb) std::memcpy(img.data() + K.prog_bytes, rowval.data(), cb);
  }

  void build_image() {
    const size_t n = K.code.size();
    // Rewrite the unified-datapath families onto (a, b, c) of fma / mad.
    // The addend reads c ^ aux: an immediate addend goes into aux with c on
    // the zero row (no constant row), a register addend has aux 0 (integer)
    // or the sign flip of a subtraction (f32). Integer subtraction needs no
    // negation: a - b = b * (-1) + a, a - imm = a * 1 + (-imm).
    std::vector<Route> route(n);
    auto is_const = [](uint8_t o) { return (o & KS_CONST_BIT) != 0; };
    auto cval = [&](uint8_t o) { return (uint32_t)K.cpool[o & 0x7F]; };
    for (size_t i = 0; i < n; i++) {
      const KsInsn& in = K.code[i];
      Route r{in.a, in.b, in.c, 0};
      if (fpu_family(in.op)) {
        if (in.op == OP_FADD || in.op == OP_FSUB) {
          uint8_t x = in.a, y = in.b;
          const uint32_t flip = in.op == OP_FSUB ? 0x80000000u : 0u;
          if (in.op == OP_FADD && is_const(x) && !is_const(y)) std::swap(x, y);  // add is commutative
          r.a = x;
          r.b = constant(0x3F800000ull, in_line(i));
          if (is_const(y)) { r.c = OPND_ZERO; r.aux = cval(y) ^ flip; }
          else { r.c = y; r.aux = flip; }
        } else if (in.op == OP_FMUL) {
          r.c = OPND_ZERO;
          r.aux = 0x80000000u;  // + (-0.0): x * y exactly rounded, signs of zero kept
        } else if (is_const(in.c)) {  // fma with an immediate addend
          r.c = OPND_ZERO;
          r.aux = cval(in.c);
        }
      } else if (imad_family(in.op)) {
        if (in.op == OP_ADD32) {
          uint8_t x = in.a, y = in.b;
          if (is_const(x) && !is_const(y)) std::swap(x, y);
          r.a = x;
          r.b = constant(1ull, in_line(i));
          if (is_const(y)) { r.c = OPND_ZERO; r.aux = cval(y); }
          else { r.c = y; r.aux = 0; }
        } else if (in.op == OP_SUB32) {
          if (is_const(in.b)) {
            r.a = in.a;
            r.b = constant(1ull, in_line(i));
            r.c = OPND_ZERO;
            r.aux = 0u - cval(in.b);
          } else {
            r.a = in.b;
            r.b = constant(0xFFFFFFFFull, in_line(i));
            if (is_const(in.a)) { r.c = OPND_ZERO; r.aux = cval(in.a); }
            else { r.c = in.a; r.aux = 0; }
          }
        } else if (in.op == OP_MUL32) {
          r.c = OPND_ZERO;
        } else if (in.op == OP_MAD32) {
          if (is_const(in.c)) { r.c = OPND_ZERO; r.aux = cval(in.c); }
        } else if (in.op == OP_MOV32) {
          if (is_const(in.a)) { r.a = r.b = r.c = OPND_ZERO; r.aux = cval(in.a); }
          else { r.b = constant(1ull, in_line(i)); r.c = OPND_ZERO; }
        }
      } else if (imm_b_op(in.op)) {
        // 32-bit logic and shifts (of either width) read b | aux
        uint8_t x = in.a, y = in.b;
        const bool commutes = in.op == OP_AND32 || in.op == OP_OR32 || in.op == OP_XOR32;
        if (commutes && is_const(x) && !is_const(y)) std::swap(x, y);
        if (is_const(y)) { r.a = x; r.b = OPND_ZERO; r.aux = cval(y); }
      }
      route[i] = r;
    }
    // Immediate multipliers. A constant row costs a warp 256 bytes of shared
    // memory, and kernels whose address arithmetic multiplies by many
    // distinct immediates fill their regions with them: when the rows would
    // pass MANY_CONST_ROWS, every unguarded mul.lo / mad.lo of a register by
    // an immediate leaves the fast path for the mid loop as DOP_MADI
    // (d = a * aux + c row) or DOP_MADII (d = a * aux + hc, an immediate
    // addend in the record's hc field, which ops without predicate operands
    // do not use), and its immediates leave the rows.
    constexpr size_t MANY_CONST_ROWS = 16;
    std::vector<uint8_t> madi(n, 0);
    std::vector<uint32_t> madi_c(n, 0);
    {
      std::vector<char> used(K.cpool.size(), 0);
      size_t rows = 0;
      for (size_t i = 0; i < n; i++) {
        const uint8_t ops[4] = {route[i].a, route[i].b, route[i].c, K.code[i].d};
        for (int p = 0; p < 4; p++)
          if (routed_width(K.code[i], p) && ops[p] != OPND_ZERO && is_const(ops[p]) && !used[ops[p] & 0x7F]) {
            used[ops[p] & 0x7F] = 1;
            rows++;
          }
      }
      if (rows > MANY_CONST_ROWS) {
        for (size_t i = 0; i < n; i++) {
          const KsInsn& in = K.code[i];
          if (in.guard != KS_NO_GUARD || (in.op != OP_MUL32 && in.op != OP_MAD32)) continue;
          uint8_t x = in.a, y = in.b;
          if (is_const(x) && !is_const(y)) std::swap(x, y);  // the product commutes
          if (is_const(x) || !is_const(y)) continue;
          Route r{x, OPND_ZERO, OPND_ZERO, cval(y)};
          if (in.op == OP_MAD32 && is_const(in.c)) {
            madi[i] = 2;
            madi_c[i] = cval(in.c);
          } else {
            madi[i] = 1;
            if (in.op == OP_MAD32) r.c = in.c;
          }
          route[i] = r;
        }
      }
    }
    // constant rows: one per constant still read from a row, two if any such
    // use is 64-bit
    std::vector<unsigned> cwidth(K.cpool.size(), 0);
    for (size_t i = 0; i < n; i++) {
      const KsInsn& in = K.code[i];
      const uint8_t ops[4] = {route[i].a, route[i].b, route[i].c, in.d};
      for (int p = 0; p < 4; p++) {
        const unsigned w = routed_width(in, p);
        if (w && ops[p] != OPND_ZERO && (ops[p] & KS_CONST_BIT))
          cwidth[ops[p] & 0x7F] = std::max(cwidth[ops[p] & 0x7F], w);
      }
    }
    std::vector<uint32_t> crow(K.cpool.size(), 0), rowval;
    for (size_t k = 0; k < K.cpool.size(); k++) {
      if (!cwidth[k]) continue;
      crow[k] = (uint32_t)rowval.size();
      rowval.push_back((uint32_t)K.cpool[k]);
      if (cwidth[k] == 64) rowval.push_back((uint32_t)(K.cpool[k] >> 32));
    }
    // one program image per layout
    for (uint32_t split = 0; split < 2; split++) resolve_image(split, route, madi, madi_c, crow, rowval);
    live_in_slots();
  }

  // The register slots that some path from the entry may read before writing
  // them (backward liveness over the program's control flow; a guarded write
  // kills nothing, since some lanes may skip it). Only these must start at 0
  // in each simulated warp; every other slot is written before it is read.
  void live_in_slots() {
    const size_t n = K.code.size();
    using Set = std::array<uint64_t, 2>;  // KS_MAX_SLOTS <= 128 bits
    auto add = [](Set& x, unsigned s, unsigned w) {
      for (unsigned k = 0; k < (w == 64 ? 2u : 1u) && s + k < KS_MAX_SLOTS; k++) x[(s + k) >> 6] |= 1ull << ((s + k) & 63);
    };
    std::vector<Set> use(n, Set{0, 0}), kill(n, Set{0, 0}), in(n + 1, Set{0, 0});
    for (size_t i = 0; i < n; i++) {
      const KsInsn& k = K.code[i];
      const uint8_t ops[3] = {k.a, k.b, k.c};
      for (int p = 0; p < 3; p++) {
        const unsigned w = row_width(k, p);
        if (w && ops[p] < KS_MAX_SLOTS) add(use[i], ops[p], w);
      }
      const unsigned wd = row_width(k, 3);
      if (wd && k.d < KS_MAX_SLOTS && k.guard == KS_NO_GUARD) add(kill[i], k.d, wd);
    }
    // successors: the next entry unless an unguarded bra or ret ends the
    // path here; a bra's target
    for (bool changed = true; changed;) {
      changed = false;
      for (size_t i = n; i-- > 0;) {
        const KsInsn& k = K.code[i];
        const bool ends = (k.op == OP_BRA || k.op == OP_RET) && k.guard == KS_NO_GUARD;
        Set out{0, 0};
        if (!ends) out = in[i + 1];
        if (k.op == OP_BRA && k.target <= n) {
          out[0] |= in[k.target][0];
          out[1] |= in[k.target][1];
        }
        const Set v{use[i][0] | (out[0] & ~kill[i][0]), use[i][1] | (out[1] & ~kill[i][1])};
        if (v != in[i]) {
          in[i] = v;
          changed = true;
        }
      }
    }
    const Set& e = n ? in[0] : in[n];
    for (int w = 0; w < 4; w++) K.live_in[w] = (uint32_t)(e[w >> 1] >> (32 * (w & 1)));
  }
};

}  // namespace

int decode_module(const char* text, size_t len, std::vector<KsKernel>* out, std::string* err) {
  try {
    Parser P(lex(text, len));
    std::vector<KernelText> kts = P.module();
    out->clear();
    for (KernelText& kt : kts) {
      for (const KsKernel& k : *out)
        if (k.name == kt.name) fail(KS_ERR_PARSE, kt.line, "kernel defined twice: " + kt.name);
      KsKernel k;
      Decoder D(kt, k);
      D.run();
      out->push_back(std::move(k));
    }
    if (out->empty()) fail(KS_ERR_PARSE, 0, "no .entry in the module");
    err->clear();
    return KS_OK;
  } catch (const Fail& f) {
    *err = f.msg;
    return f.code;
  } catch (const std::exception& e) {
    *err = e.what();
    return KS_ERR_PARSE;
  }
}

}  // namespace ks
