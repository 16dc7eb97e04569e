// SDF delay statements -> the per-instance delay tables and interconnect delays of
// the simulator (host code).
//
// GATSPI (Section 3, Fig. 4) translates SDF IOPATH and COND statements into a 2-D
// array per instance: a row per switching pin, input edge and output edge (row =
// 4 * pin + 2 * e_in + e_out, RISE = 0, FALL = 1), a column per combination of the
// other pins' values (in pin order, the first one most significant), so that the
// conditional delay of an arc is one lookup and no calibration run is needed.
//
// Rules (the page gives the arrays, not the parser):
//   - (IOPATH (posedge P) Y r f) sets pin P's rows with e_in = RISE, (negedge P)
//     those with e_in = FALL, a bare P both; r is the output-rise delay and f the
//     output-fall delay (one value serves both); an empty () is no arc (NO_ARC);
//   - an unconditional IOPATH sets every column; (COND expr (IOPATH ...)) sets the
//     columns where expr holds for the other pins' values, over the unconditional
//     statements whatever the order; where several hold, the last one written wins;
//   - min:typ:max triples give typ; values are converted from the file's TIMESCALE
//     (1 ns when absent) to the simulator's unit exactly and rounded to the nearest
//     integer, halves up; negative values are rejected;
//   - (INTERCONNECT src inst/pin r f) gives that pin's wire delays; others stay 0;
//   - table entries no statement sets stay NO_ARC.
// Conditions are Verilog expressions (== === != !== ! ~ & | ^ && || and
// parentheses) over the other pins, with the literals 0, 1, 1'b0, 1'b1, 'b0, 'b1.
#include <cctype>
#include <cstdio>
#include <cstring>
#include <string>
#include <string_view>
#include <unordered_map>
#include <vector>

#include "gatspi.h"

void gatspi_set_last_error(const char *msg);

namespace {

struct SdfFail {
    std::string msg;
};

[[noreturn]] void sdf_fail(const std::string &m) { throw SdfFail{m}; }

// ---- S-expression tree -----------------------------------------------------------

struct Node {
    bool list;
    std::string_view atom;     // atoms
    int first = -1, count = 0; // lists: children in kids[first .. first + count)
};

struct Tree {
    std::vector<Node> nodes;
    std::vector<int> kids;
    const Node &kid(const Node &n, int k) const { return nodes[kids[n.first + k]]; }
    bool is(const Node &n, const char *head) const {
        return n.list && n.count > 0 && !kid(n, 0).list && kid(n, 0).atom == head;
    }
};

constexpr size_t kMaxListDepth = 1000;

Tree parse_tree(std::string_view s) {
    Tree t;
    t.nodes.reserve(s.size() / 4 + 16);
    t.kids.reserve(s.size() / 4 + 16);
    std::vector<int> pending;   // children of the open lists, innermost last
    std::vector<size_t> marks;  // where each open list's children start in pending
    marks.push_back(0);
    size_t i = 0;
    const size_t n = s.size();
    while (i < n) {
        const char c = s[i];
        if (std::isspace((unsigned char)c)) {
            ++i;
        } else if (c == '(') {
            // lists are walked recursively later (flatten): bound their depth, far
            // beyond any SDF statement (a few levels; conditions stop at 48 anyway)
            if (marks.size() > kMaxListDepth) sdf_fail("lists nested too deeply at byte " + std::to_string(i));
            marks.push_back(pending.size());
            ++i;
        } else if (c == ')') {
            if (marks.size() == 1) sdf_fail("unbalanced parentheses at byte " + std::to_string(i));
            const size_t m = marks.back();
            marks.pop_back();
            Node nd{true, {}, (int)t.kids.size(), (int)(pending.size() - m)};
            t.kids.insert(t.kids.end(), pending.begin() + (long)m, pending.end());
            pending.resize(m);
            t.nodes.push_back(nd);
            pending.push_back((int)t.nodes.size() - 1);
            ++i;
        } else {
            // a quoted string runs to the next quote, wherever it is; a quote with none
            // after it starts an ordinary atom, which runs to a space or a parenthesis
            size_t j = c == '"' ? s.find('"', i + 1) : std::string_view::npos;
            if (j != std::string_view::npos) {
                ++j;
            } else {
                j = i;
                while (j < n && !std::isspace((unsigned char)s[j]) && s[j] != '(' && s[j] != ')') ++j;
            }
            t.nodes.push_back(Node{false, s.substr(i, j - i)});
            pending.push_back((int)t.nodes.size() - 1);
            i = j;
        }
    }
    if (marks.size() != 1 || pending.size() != 1) sdf_fail("unbalanced parentheses");
    Node root{true, {}, (int)t.kids.size(), 1};
    t.kids.push_back(pending[0]);
    t.nodes.push_back(root);
    return t;
}

// ---- conditions ------------------------------------------------------------------

// Operators and operands of a condition, in postfix order.
enum Op : int { kVar = 0, kConst, kNot, kAnd, kOr, kBitAnd, kBitOr, kXor, kEq, kNe };

struct Cond {
    static constexpr int kStack = 256;   // operands eval can hold at once
    std::vector<int> code;   // pairs (op, arg)
    bool names(int pin) const {
        for (size_t k = 0; k < code.size(); k += 2)
            if (code[k] == kVar && code[k + 1] == pin) return true;
        return false;
    }
    // Most operands pending at once while evaluating: the parser refuses a condition
    // that needs more than kStack (nesting is bounded, but each level can leave one
    // operand pending per binary precedence level).
    int stack_depth() const {
        int sp = 0, most = 0;
        for (size_t k = 0; k < code.size(); k += 2) {
            const int op = code[k];
            sp += (op == kVar || op == kConst) ? 1 : (op == kNot ? 0 : -1);
            most = sp > most ? sp : most;
        }
        return most;
    }
    int eval(const int *val) const {
        int st[kStack];
        st[0] = 0;
        int sp = 0;
        for (size_t k = 0; k < code.size(); k += 2) {
            const int op = code[k];
            if (op == kVar) {
                st[sp++] = val[code[k + 1]];
            } else if (op == kConst) {
                st[sp++] = code[k + 1];
            } else if (op == kNot) {
                st[sp - 1] = 1 - st[sp - 1];
            } else {
                const int b = st[--sp], a = st[sp - 1];
                int r = 0;
                switch (op) {
                    case kAnd: r = (a && b); break;
                    case kOr: r = (a || b); break;
                    case kBitAnd: r = a & b; break;
                    case kBitOr: r = a | b; break;
                    case kXor: r = a ^ b; break;
                    case kEq: r = (a == b); break;
                    default: r = (a != b); break;
                }
                st[sp - 1] = r;
            }
        }
        return st[0];
    }
};

// Recursive-descent parser over the condition's tokens (Verilog precedence:
// unary, equality, &, ^, |, &&, ||).
struct CondParser {
    std::vector<std::string> tok;
    size_t k = 0;
    const std::vector<std::string> *pins = nullptr;
    Cond out;
    int depth = 0;

    void lex(const std::string &s) {
        size_t i = 0;
        while (i < s.size()) {
            const char c = s[i];
            if (std::isspace((unsigned char)c)) {
                ++i;
                continue;
            }
            static const char *ops[] = {"===", "!==", "==", "!=", "&&", "||"};
            bool done = false;
            for (const char *op : ops) {
                const size_t L = std::strlen(op);
                if (s.compare(i, L, op) == 0) {
                    tok.emplace_back(op);
                    i += L;
                    done = true;
                    break;
                }
            }
            if (done) continue;
            if (std::strchr("!~&|^()", c)) {
                tok.emplace_back(1, c);
                ++i;
            } else if (std::isdigit((unsigned char)c) || c == '\'') {
                size_t j = i;
                while (j < s.size() && (std::isalnum((unsigned char)s[j]) || s[j] == '\'')) ++j;
                tok.push_back(s.substr(i, j - i));
                i = j;
            } else if (std::isalpha((unsigned char)c) || c == '_') {
                size_t j = i;
                while (j < s.size() &&
                       (std::isalnum((unsigned char)s[j]) || s[j] == '_' || s[j] == '[' || s[j] == ']' || s[j] == '.' ||
                        s[j] == '\\'))
                    ++j;
                tok.push_back(s.substr(i, j - i));
                i = j;
            } else {
                sdf_fail("bad character in condition: " + s);
            }
        }
    }
    const std::string *peek() const { return k < tok.size() ? &tok[k] : nullptr; }
    void emit(int op, int arg = 0) {
        out.code.push_back(op);
        out.code.push_back(arg);
    }
    void binary(int level) {
        static const std::vector<std::vector<std::pair<const char *, int>>> table = {
            {{"||", kOr}}, {{"&&", kAnd}}, {{"|", kBitOr}}, {{"^", kXor}}, {{"&", kBitAnd}},
            {{"==", kEq}, {"===", kEq}, {"!=", kNe}, {"!==", kNe}}};
        if (level == (int)table.size()) {
            unary();
            return;
        }
        binary(level + 1);
        for (;;) {
            const std::string *t = peek();
            int op = -1;
            if (t)
                for (auto &e : table[level])
                    if (*t == e.first) op = e.second;
            if (op < 0) return;
            ++k;
            binary(level + 1);
            emit(op);
        }
    }
    void unary() {
        if (++depth > 48) sdf_fail("condition nested too deeply");
        const std::string *t = peek();
        if (!t) sdf_fail("truncated condition");
        if (*t == "!" || *t == "~") {
            ++k;
            unary();
            emit(kNot);
        } else if (*t == "(") {
            ++k;
            binary(0);
            if (!peek() || *peek() != ")") sdf_fail("unbalanced condition");
            ++k;
        } else {
            ++k;
            const size_t quote = t->find('\'');
            if (quote != std::string::npos) {
                // a one-bit binary literal, sized or not: digits, 'b or 'B, then 0 or 1
                bool lit = t->size() == quote + 3 && ((*t)[quote + 1] == 'b' || (*t)[quote + 1] == 'B') &&
                           (t->back() == '0' || t->back() == '1');
                for (size_t u = 0; u < quote; ++u) lit = lit && std::isdigit((unsigned char)(*t)[u]);
                if (!lit) sdf_fail("bad literal " + *t);
                emit(kConst, t->back() - '0');
            } else if (*t == "0" || *t == "1") {
                emit(kConst, (*t)[0] - '0');
            } else {
                int pin = -1;
                for (size_t q = 0; q < pins->size(); ++q)
                    if ((*pins)[q] == *t) pin = (int)q;
                if (pin < 0) sdf_fail("condition names " + *t + ", not a pin of the cell");
                emit(kVar, pin);
            }
        }
        --depth;
    }
};

// ---- values ----------------------------------------------------------------------

long long file_scale_fs(std::string s) {
    size_t d = 0;
    while (d < s.size() && (std::isdigit((unsigned char)s[d]) || s[d] == '.')) ++d;
    std::string num = s.substr(0, d), unit = s.substr(d);
    while (!num.empty() && (num.back() == '0' || num.back() == '.') && num.find('.') != std::string::npos)
        num.pop_back();
    long long m = 0;
    if (num == "1") m = 1;
    else if (num == "10") m = 10;
    else if (num == "100") m = 100;
    else sdf_fail("bad TIMESCALE " + s);
    static const std::pair<const char *, long long> units[] = {{"s", 1000000000000000ll}, {"ms", 1000000000000ll},
                                                               {"us", 1000000000ll},      {"ns", 1000000ll},
                                                               {"ps", 1000ll},            {"fs", 1ll}};
    for (auto &u : units)
        if (unit == u.first) return m * u.second;
    sdf_fail("bad TIMESCALE " + s);
}

// A decimal number times file_fs / unit_fs, rounded to the nearest integer (halves up).
int32_t convert(std::string_view v, long long file_fs, long long unit_fs) {
    __int128 mant = 0;
    int exp10 = 0, digits = 0;
    size_t i = 0;
    bool neg = false;
    if (i < v.size() && (v[i] == '+' || v[i] == '-')) neg = v[i++] == '-';
    bool dot = false, any = false;
    for (; i < v.size(); ++i) {
        const char c = v[i];
        if (c == '.' && !dot) {
            dot = true;
        } else if (std::isdigit((unsigned char)c)) {
            any = true;
            // at most 20 significant digits, so that mant * file_fs (< 10^20 * 10^17)
            // fits the 128-bit arithmetic; zeros beyond them are exact (a power of ten),
            // any other digit is refused rather than dropped
            if (digits < 20) {
                mant = mant * 10 + (c - '0');
                if (mant != 0) ++digits;
                if (dot) --exp10;
            } else if (c != '0') {
                sdf_fail("more than 20 significant digits: " + std::string(v));
            } else if (!dot) {
                ++exp10;
            }
        } else {
            break;
        }
    }
    if (i < v.size() && (v[i] == 'e' || v[i] == 'E')) {
        ++i;
        bool eneg = false;
        if (i < v.size() && (v[i] == '+' || v[i] == '-')) eneg = v[i++] == '-';
        int e = 0;
        bool edig = false;
        for (; i < v.size() && std::isdigit((unsigned char)v[i]); ++i) {
            edig = true;
            if (e < 1000) e = e * 10 + (v[i] - '0');
        }
        if (!edig) sdf_fail("bad number " + std::string(v));
        exp10 += eneg ? -e : e;
    }
    if (!any || i != v.size()) sdf_fail("bad number " + std::string(v));
    if (neg && mant != 0) sdf_fail("negative delay " + std::string(v));
    // value = mant * 10^exp10 * file_fs / unit_fs = num / den, exactly, in unsigned
    // 128-bit arithmetic: num < 10^20 * 10^17 < 2^123 to start with
    using u128 = unsigned __int128;
    u128 num = (u128)mant * (u128)file_fs, den = (u128)unit_fs;
    for (; exp10 > 0; --exp10) {
        num *= 10;
        if (num > ((u128)1 << 100)) sdf_fail("delay too large: " + std::string(v));
    }
    for (; exp10 < 0; ++exp10) {
        if (den > 2 * num) return 0;   // below one half, and every further 10 makes it smaller
        den *= 10;                     // den <= 2 num < 2^124 before, so < 2^128 after
    }
    // nearest integer, halves up: the quotient, plus one when 2 * rem >= den
    const u128 q = num / den, rem = num - q * den;
    const u128 r = q + (rem >= den - rem ? 1 : 0);
    if (r >= (u128)GATSPI_NO_ARC) sdf_fail("delay too large: " + std::string(v));
    return (int32_t)r;
}

int32_t value_of(const Tree &t, const Node &n, long long file_fs, long long unit_fs) {
    if (!n.list) sdf_fail("delay value must be parenthesised: " + std::string(n.atom));
    if (n.count == 0) return GATSPI_NO_ARC;
    if (n.count != 1 || t.kid(n, 0).list) sdf_fail("bad delay value");
    std::string_view v = t.kid(n, 0).atom;
    const size_t c1 = v.find(':');
    if (c1 != std::string_view::npos) {
        const size_t c2 = v.find(':', c1 + 1);
        if (c2 == std::string_view::npos || v.find(':', c2 + 1) != std::string_view::npos)
            sdf_fail("bad delay value " + std::string(v));
        v = v.substr(c1 + 1, c2 - c1 - 1);   // typ
    }
    return convert(v, file_fs, unit_fs);
}

void rise_fall(const Tree &t, const Node &st, int first, long long file_fs, long long unit_fs, int32_t &r,
               int32_t &f) {
    if (st.count <= first) sdf_fail("statement without delay values");
    r = value_of(t, t.kid(st, first), file_fs, unit_fs);
    f = st.count > first + 1 ? value_of(t, t.kid(st, first + 1), file_fs, unit_fs) : r;
}

void flatten(const Tree &t, const Node &n, std::string &s) {
    if (!n.list) {
        s.append(n.atom);
        s.push_back(' ');
        return;
    }
    s.append("( ");
    for (int k = 0; k < n.count; ++k) flatten(t, t.kid(n, k), s);
    s.append(") ");
}

struct Annotator {
    const gatspi_sdf_design *d;
    std::vector<std::vector<std::string>> pins;   // per type
    std::vector<long long> pin_first;
    std::unordered_map<std::string_view, int> inst;
    std::unordered_map<std::string, Cond> cond_cache;   // (cell type, condition text) -> parsed
    long long file_fs = 1000000;

    void iopath(const Tree &t, const Node &st, int g, const Cond *cond, int32_t *dly) {
        const int ty = d->gate_type[g];
        const auto &pn = pins[ty];
        const int n = (int)pn.size();
        if (st.count < 4) sdf_fail("short IOPATH");
        const Node &port = t.kid(st, 1), &outp = t.kid(st, 2);
        if (outp.list || outp.atom != d->out_pin) sdf_fail("IOPATH to a pin that is not the output");
        int edges = 3;   // bit 0: RISE input edge, bit 1: FALL
        std::string_view name;
        if (port.list) {
            if (port.count != 2 || t.kid(port, 0).list || t.kid(port, 1).list) sdf_fail("bad IOPATH port");
            const std::string_view e = t.kid(port, 0).atom;
            if (e == "posedge") edges = 1;
            else if (e == "negedge") edges = 2;
            else sdf_fail("bad edge " + std::string(e));
            name = t.kid(port, 1).atom;
        } else {
            name = port.atom;
        }
        int pin = -1;
        for (int q = 0; q < n; ++q)
            if (pn[q] == name) pin = q;
        if (pin < 0) sdf_fail("no pin " + std::string(name));
        if (cond && cond->names(pin)) sdf_fail("a condition names the switching pin " + std::string(name));
        int32_t r, f;
        rise_fall(t, st, 3, file_fs, d->unit_fs, r, f);
        const int cols = 1 << (n - 1);
        int32_t *D = dly + d->gate_dly_off[g];
        int val[8] = {0};
        for (int c = 0; c < cols; ++c) {
            if (cond) {
                for (int q = 0, k = 0; q < n; ++q)
                    if (q != pin) val[q] = (c >> (n - 2 - k++)) & 1;
                if (!cond->eval(val)) continue;
            }
            for (int e_in = 0; e_in < 2; ++e_in)
                if (edges & (1 << e_in)) {
                    D[(4 * pin + 2 * e_in + 0) * cols + c] = r;
                    D[(4 * pin + 2 * e_in + 1) * cols + c] = f;
                }
        }
    }

    void run(const Tree &t, int32_t *dly, int32_t *wr, int32_t *wf) {
        const Node &root = t.kid(t.nodes.back(), 0);
        if (!t.is(root, "DELAYFILE")) sdf_fail("not a DELAYFILE");
        for (int k = 1; k < root.count; ++k) {
            const Node &it = t.kid(root, k);
            if (t.is(it, "TIMESCALE")) {
                std::string s;
                for (int q = 1; q < it.count; ++q)
                    if (!t.kid(it, q).list) s.append(t.kid(it, q).atom);
                file_fs = file_scale_fs(s);
            }
        }
        std::vector<int> conds;
        for (int k = 1; k < root.count; ++k) {
            const Node &cell = t.kid(root, k);
            if (!t.is(cell, "CELL")) continue;
            std::string_view celltype, iname;
            bool has_inst = false;
            std::vector<int> stmts;
            for (int q = 1; q < cell.count; ++q) {
                const Node &part = t.kid(cell, q);
                if (t.is(part, "CELLTYPE")) {
                    if (part.count < 2 || t.kid(part, 1).list) sdf_fail("bad CELLTYPE");
                    // the name without the quotes around it (every leading and trailing one)
                    celltype = t.kid(part, 1).atom;
                    const size_t a = celltype.find_first_not_of('"'), b = celltype.find_last_not_of('"');
                    celltype = a == std::string_view::npos ? std::string_view() : celltype.substr(a, b - a + 1);
                } else if (t.is(part, "INSTANCE")) {
                    if (part.count > 1) {
                        iname = t.kid(part, 1).atom;
                        has_inst = !iname.empty();
                    }
                } else if (t.is(part, "DELAY")) {
                    for (int b = 1; b < part.count; ++b) {
                        const Node &block = t.kid(part, b);
                        if (!t.is(block, "ABSOLUTE")) sdf_fail("only ABSOLUTE delays are read");
                        for (int s = 1; s < block.count; ++s) stmts.push_back(t.kids[block.first + s]);
                    }
                }
            }
            int g = -1;
            if (has_inst) {
                auto f = inst.find(iname);
                if (f == inst.end()) sdf_fail("unknown instance " + std::string(iname));
                g = f->second;
                if (celltype != d->type_names[d->gate_type[g]])
                    sdf_fail("instance " + std::string(iname) + " is not a " + std::string(celltype));
            }
            conds.clear();
            for (int s : stmts) {
                const Node &st = t.nodes[s];
                if (t.is(st, "INTERCONNECT")) {
                    if (st.count < 4 || t.kid(st, 2).list) sdf_fail("bad INTERCONNECT");
                    const std::string_view dst = t.kid(st, 2).atom;
                    const size_t slash = dst.rfind('/');
                    if (slash == std::string_view::npos) sdf_fail("INTERCONNECT destination is not inst/pin");
                    auto f = inst.find(dst.substr(0, slash));
                    if (f == inst.end()) sdf_fail("unknown instance " + std::string(dst.substr(0, slash)));
                    const int dg = f->second;
                    const auto &pn = pins[d->gate_type[dg]];
                    int pin = -1;
                    for (size_t q = 0; q < pn.size(); ++q)
                        if (pn[q] == dst.substr(slash + 1)) pin = (int)q;
                    if (pin < 0) sdf_fail("no pin " + std::string(dst));
                    int32_t r, fl;
                    rise_fall(t, st, 3, file_fs, d->unit_fs, r, fl);
                    const long long e = (long long)d->fanin_off[dg] + pin;
                    if (wr) wr[e] = r;
                    if (wf) wf[e] = fl;
                } else if (t.is(st, "IOPATH")) {
                    if (g < 0) sdf_fail("IOPATH outside an instance");
                    iopath(t, st, g, nullptr, dly);
                } else if (t.is(st, "COND")) {
                    if (g < 0) sdf_fail("COND outside an instance");
                    conds.push_back(s);
                } else {
                    sdf_fail("unsupported statement");
                }
            }
            for (int s : conds) {   // after every unconditional statement, in file order
                const Node &st = t.nodes[s];
                const Node &body = t.kid(st, st.count - 1);
                if (st.count < 3 || !t.is(body, "IOPATH")) sdf_fail("COND without IOPATH");
                int from = 1;
                if (!t.kid(st, 1).list && !t.kid(st, 1).atom.empty() && t.kid(st, 1).atom.front() == '"') from = 2;
                std::string text = std::to_string(d->gate_type[g]) + "|";
                for (int q = from; q < st.count - 1; ++q) flatten(t, t.kid(st, q), text);
                auto hit = cond_cache.find(text);
                if (hit == cond_cache.end()) {
                    CondParser cp;
                    cp.pins = &pins[d->gate_type[g]];
                    cp.lex(text.substr(text.find('|') + 1));
                    cp.binary(0);
                    if (cp.k != cp.tok.size()) sdf_fail("bad condition: " + text);
                    if (cp.out.stack_depth() > Cond::kStack) sdf_fail("condition too long: " + text);
                    hit = cond_cache.emplace(std::move(text), std::move(cp.out)).first;
                }
                iopath(t, body, g, &hit->second, dly);
            }
        }
    }
};

thread_local char g_sdf_msg[512];

}  // namespace

extern "C" gatspi_status gatspi_sdf_annotate(const gatspi_sdf_design *d, const char *text, size_t len,
                                             int32_t *dly_data, int32_t *wire_rise, int32_t *wire_fall) {
    auto err = [](gatspi_status s, const char *m) {
        gatspi_set_last_error(m);
        return s;
    };
    if (!d || (!text && len) || !dly_data) return err(GATSPI_EINVAL, "design, text and dly_data are required");
    if (d->num_types < 0 || d->num_gates < 0 || d->unit_fs < 1 || d->dly_len < 0 || !d->out_pin)
        return err(GATSPI_EINVAL, "bad design sizes");
    if (d->num_gates > 0 && (!d->type_names || !d->type_num_pins || !d->pin_names || !d->gate_type ||
                             !d->instance_names || !d->fanin_off || !d->gate_dly_off))
        return err(GATSPI_EINVAL, "every array of gatspi_sdf_design is required");
    try {
        Annotator a;
        a.d = d;
        a.pins.resize(d->num_types);
        long long off = 0;
        for (int ty = 0; ty < d->num_types; ++ty) {
            const int n = d->type_num_pins[ty];
            if (n < 1 || n > GATSPI_MAX_PINS) sdf_fail("type " + std::to_string(ty) + ": bad pin count");
            for (int q = 0; q < n; ++q) a.pins[ty].emplace_back(d->pin_names[off + q]);
            off += n;
        }
        a.inst.reserve((size_t)d->num_gates * 2);
        for (int g = 0; g < d->num_gates; ++g) {
            const int ty = d->gate_type[g];
            if (ty < 0 || ty >= d->num_types) sdf_fail("gate " + std::to_string(g) + ": bad type");
            const int n = d->type_num_pins[ty];
            if (d->gate_dly_off[g] < 0 || d->gate_dly_off[g] + 4ll * n * (1 << (n - 1)) > d->dly_len)
                sdf_fail("gate " + std::to_string(g) + ": delay table out of range");
            if (!a.inst.emplace(std::string_view(d->instance_names[g]), g).second)
                sdf_fail(std::string("duplicate instance name ") + d->instance_names[g]);
        }
        // every table starts as "no arc", everything else as 0; wires as 0
        std::memset(dly_data, 0, sizeof(int32_t) * (size_t)d->dly_len);
        for (int g = 0; g < d->num_gates; ++g) {
            const int n = d->type_num_pins[d->gate_type[g]];
            int32_t *D = dly_data + d->gate_dly_off[g];
            for (long long k = 0; k < 4ll * n * (1 << (n - 1)); ++k) D[k] = GATSPI_NO_ARC;
        }
        const long long E = d->num_gates > 0 ? d->fanin_off[d->num_gates] : 0;
        if (wire_rise) std::memset(wire_rise, 0, sizeof(int32_t) * (size_t)E);
        if (wire_fall) std::memset(wire_fall, 0, sizeof(int32_t) * (size_t)E);
        const Tree t = parse_tree(std::string_view(text ? text : "", len));
        a.run(t, dly_data, wire_rise, wire_fall);
    } catch (const SdfFail &f) {
        std::snprintf(g_sdf_msg, sizeof g_sdf_msg, "SDF: %s", f.msg.c_str());
        return err(GATSPI_EINVAL, g_sdf_msg);
    } catch (const std::bad_alloc &) {
        return err(GATSPI_ENOMEM, "SDF: out of host memory");
    }
    gatspi_set_last_error("");
    return GATSPI_OK;
}
