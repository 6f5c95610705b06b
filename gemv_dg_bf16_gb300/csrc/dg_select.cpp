// dg_select.cpp -- per-device shape table: parse, identity checks, lookup.
//
// mstar PR #1104, "What changed": one per-device table keyed by op, size and
// the decode bucket's rows, each entry keeping every candidate's time and
// parameters beside the choice; without a table the compiled defaults stay.
// Strata PR #1297, "The second commit: the seam rework": the table carries an
// identity (architecture, runtime, build) plus a kernel-selection-space token,
// refuses when any of them differs or when a dispatch knob reroutes the
// launch, prints one stderr line and keeps the defaults; one rows list feeds
// the parser, the launchers and the sweep.
// "Decode optimization round 3", "Retained change 2": lookups pad M up to the
// next listed bucket and never fall back to a nearest row.
#include <atomic>
#include <cctype>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <map>
#include <memory>
#include <mutex>
#include <sstream>
#include <string>
#include <tuple>
#include <vector>

#include "dg_internal.h"
#include "dg_rows.h"

namespace dg {
namespace {

// ------------------------------------------------------------------ JSON subset
struct JVal {
    enum Kind { Null, Bool, Num, Str, Arr, Obj } kind = Null;
    double num = 0;
    bool b = false;
    std::string str;
    std::vector<JVal> arr;
    std::vector<std::pair<std::string, JVal>> obj;
    const JVal* get(const char* k) const
    {
        for (auto& kv : obj)
            if (kv.first == k) return &kv.second;
        return nullptr;
    }
};

struct JParser {
    const char* p;
    const char* end;
    std::string err;
    void ws()
    {
        while (p < end && std::isspace(static_cast<unsigned char>(*p))) ++p;
    }
    bool lit(const char* s)
    {
        size_t n = std::strlen(s);
        if (static_cast<size_t>(end - p) >= n && std::strncmp(p, s, n) == 0) {
            p += n;
            return true;
        }
        return false;
    }
    bool parse(JVal& v, int depth = 0)
    {
        if (depth > 32) return fail("nesting too deep");
        ws();
        if (p >= end) return fail("unexpected end");
        if (*p == '{') {
            ++p;
            v.kind = JVal::Obj;
            ws();
            if (p < end && *p == '}') { ++p; return true; }
            for (;;) {
                ws();
                JVal key;
                if (p >= end || *p != '"' || !parse_str(key.str)) return fail("expected key");
                ws();
                if (p >= end || *p != ':') return fail("expected ':'");
                ++p;
                JVal val;
                if (!parse(val, depth + 1)) return false;
                v.obj.emplace_back(key.str, std::move(val));
                ws();
                if (p < end && *p == ',') { ++p; continue; }
                if (p < end && *p == '}') { ++p; return true; }
                return fail("expected ',' or '}'");
            }
        }
        if (*p == '[') {
            ++p;
            v.kind = JVal::Arr;
            ws();
            if (p < end && *p == ']') { ++p; return true; }
            for (;;) {
                JVal val;
                if (!parse(val, depth + 1)) return false;
                v.arr.push_back(std::move(val));
                ws();
                if (p < end && *p == ',') { ++p; continue; }
                if (p < end && *p == ']') { ++p; return true; }
                return fail("expected ',' or ']'");
            }
        }
        if (*p == '"') {
            v.kind = JVal::Str;
            return parse_str(v.str);
        }
        if (lit("true")) { v.kind = JVal::Bool; v.b = true; return true; }
        if (lit("false")) { v.kind = JVal::Bool; v.b = false; return true; }
        if (lit("null")) { v.kind = JVal::Null; return true; }
        char* q = nullptr;
        std::string tmp(p, std::min<size_t>(static_cast<size_t>(end - p), 64));
        double d = std::strtod(tmp.c_str(), &q);
        if (q == tmp.c_str()) return fail("bad value");
        p += (q - tmp.c_str());
        v.kind = JVal::Num;
        v.num = d;
        return true;
    }
    bool parse_str(std::string& out)
    {
        ++p;  // opening quote
        while (p < end && *p != '"') {
            if (*p == '\\') {
                ++p;
                if (p >= end) return fail("bad escape");
                char c = *p;
                out.push_back(c == 'n' ? '\n' : c == 't' ? '\t' : c);
            } else {
                out.push_back(*p);
            }
            ++p;
        }
        if (p >= end) return fail("unterminated string");
        ++p;
        return true;
    }
    bool fail(const char* m)
    {
        if (err.empty()) err = m;
        return false;
    }
};

// ------------------------------------------------------------------ table state
struct Entry {
    dg_choice choice;
};
using Key = std::tuple<int, int, int, int>;   // op, bucket M, N, K

std::mutex g_tmu;
std::map<Key, Entry> g_table;
std::string g_table_path;

const char* op_name(int op)
{
    switch (op) {
    case DG_OP_GEMV_BF16: return "gemv_bf16";
    case DG_OP_GATE_UP_SILU: return "gate_up_silu";
    case DG_OP_HEAD_FP8_ARGMAX: return "head_fp8_argmax";
    case DG_OP_MOE_W1: return "moe_w1_silu";
    case DG_OP_MOE_W2: return "moe_w2";
    case DG_OP_GEMV_A8W8: return "gemv_a8w8";
    default: return nullptr;
    }
}

int op_from_name(const std::string& s)
{
    for (int op = 0; op < DG_OP_COUNT; ++op)
        if (s == op_name(op)) return op;
    return -1;
}

bool valid_bucket(int m)
{
    static const int rows[] = {DG_ROWS_BUCKETS(DG_ROWS_AS_LIST)};
    for (int r : rows)
        if (r == m) return true;
    return false;
}

// Returns "" when the choice is acceptable for the op, else the reason.
std::string check_choice(int op, const dg_choice& c)
{
    if (op == DG_OP_GEMV_A8W8 && c.variant != DG_VAR_TC) return "the A8W8 linear runs on the tensor cores only";
    if (c.variant == DG_VAR_TC) {
        if (c.params[0] != 0 && (c.params[0] < 2 || c.params[0] > 8)) return "pipeline stages must be 2..8";
        const bool dense = op == DG_OP_GEMV_BF16 || op == DG_OP_GATE_UP_SILU || op == DG_OP_GEMV_A8W8;
        if (dense && c.params[1] != 0 && c.params[1] != 1)
            return op == DG_OP_GEMV_A8W8 ? "A8W8 quantisation launch flag must be 0 or 1"
                                         : "tensor-core K-split rule must be 0 or 1";
        for (int i = dense ? 2 : 1; i < 6; ++i)
            if (c.params[i] != 0) return "unused tensor-core parameter set";
        return "";
    }
    if (c.variant == DG_VAR_MMA) {
        if (op != DG_OP_GEMV_BF16 && op != DG_OP_GATE_UP_SILU) return "no warp-level tensor-core variant for this op";
        const int ks = c.params[0], wpc = c.params[1], u = c.params[3];
        if ((ks != 0 && ks != 1 && ks != 2 && ks != 4 && ks != 8) || (wpc != 0 && wpc != 4 && wpc != 8) ||
            c.params[2] < 0 || (u != 0 && u != 2 && u != 4 && u != 8) || c.params[4] != 0 || c.params[5] != 0)
            return "warp-level tensor-core parameters out of range";
        if (ks > (wpc ? wpc : 8)) return "K-split warps must divide warps per CTA";
        return "";
    }
    if (c.variant == DG_VAR_CC_BULK) {
        if (op != DG_OP_GEMV_BF16 && op != DG_OP_GATE_UP_SILU && op != DG_OP_HEAD_FP8_ARGMAX)
            return "no bulk-staged variant for this op";
        if (c.params[0] != 0 || c.params[1] < 0 || c.params[1] == 1 || c.params[1] > 32 || c.params[2] < 0 ||
            c.params[2] > 2)
            return "bulk-staged parameters out of range";
        return "";
    }
    if (c.variant != DG_VAR_CC_WARP) return "variant not in this build's selection space";
    const int R = c.params[0], wpc = c.params[1];
    if (op == DG_OP_MOE_W1 || op == DG_OP_MOE_W2) {
        if (R != 0 && R != 4) return "MoE rows per warp must be 4";
        const int mt = c.params[4];
        if (mt != 0 && mt != 1 && mt != 2 && mt != 4 && mt != 8) return "MoE pairs per pass must be 1, 2, 4 or 8";
        if (c.params[5] != 0 && c.params[5] != kMoeOrderUnits && c.params[5] != kMoeOrderRange)
            return "MoE work order must be 0, 1 or 2";
        if (c.params[5] == kMoeOrderRange && ((wpc != 4 && wpc != 8) || c.params[2] > 4 || c.params[3] != 0))
            return "MoE row-range parameters out of range";
    } else if (R != 1 && R != 2 && R != 4 && R != 8) {
        return "rows per warp must be 1, 2, 4 or 8";
    }
    if (op == DG_OP_GATE_UP_SILU && R < 2) return "gate/up needs an even rows-per-warp";
    if (wpc < 1 || wpc > 8) return "warps per CTA must be 1..8";
    for (int i = 2; i < 6; ++i)
        if (c.params[i] < 0) return "negative parameter";
    if (op != DG_OP_MOE_W1 && op != DG_OP_MOE_W2) {
        const int ks = c.params[3];
        if (ks != 0 && ks != 1 && ks != 2 && ks != 4 && ks != 8) return "K-split warps must be 1, 2, 4 or 8";
        if (ks > 1 && wpc % ks != 0) return "K-split warps must divide warps per CTA";
        if (c.params[4] != 0) return "unused parameter set";
    }
    return "";
}

bool parse_choice(const JVal* v, dg_choice& c)
{
    if (!v || v->kind != JVal::Obj) return false;
    std::memset(&c, 0, sizeof c);
    const JVal* var = v->get("variant");
    const JVal* par = v->get("params");
    if (!var || var->kind != JVal::Num || !par || par->kind != JVal::Arr || par->arr.size() > 6)
        return false;
    c.variant = static_cast<int32_t>(var->num);
    for (size_t i = 0; i < par->arr.size(); ++i) {
        if (par->arr[i].kind != JVal::Num) return false;
        c.params[i] = static_cast<int32_t>(par->arr[i].num);
    }
    return true;
}

const char* force_knob()
{
    const char* k = std::getenv("DG_FORCE_VARIANT");
    return (k && *k) ? k : nullptr;
}

// Parse + check.  On success fills `out` and returns DG_OK.
dg_status load_impl(const char* path, const char* arch, int drv, int rt, std::map<Key, Entry>* out,
                    std::string& reason)
{
    if (!path) {
        reason = "no path";
        return DG_ERR_INVALID_ARG;
    }
    std::ifstream f(path, std::ios::binary);
    if (!f) {
        reason = std::string("cannot read ") + path;
        return DG_ERR_TABLE_REFUSED;
    }
    std::stringstream ss;
    ss << f.rdbuf();
    const std::string text = ss.str();
    JParser jp{text.data(), text.data() + text.size(), {}};
    JVal root;
    if (!jp.parse(root) || root.kind != JVal::Obj) {
        reason = "not a valid table (" + (jp.err.empty() ? std::string("not an object") : jp.err) + ")";
        return DG_ERR_TABLE_REFUSED;
    }
    const JVal* fmt = root.get("format");
    if (!fmt || fmt->kind != JVal::Str || fmt->str != "libdecodegemm-table") {
        reason = "not a libdecodegemm table";
        return DG_ERR_TABLE_REFUSED;
    }
    const JVal* id = root.get("identity");
    if (!id || id->kind != JVal::Obj) {
        reason = "table has no identity header";
        return DG_ERR_TABLE_REFUSED;
    }
    const JVal* space = id->get("selection_space");
    if (!space) {
        reason = "made before the kernel selection space was tracked - the kernels have changed since: run the sweep again";
        return DG_ERR_TABLE_REFUSED;
    }
    if (space->kind != JVal::Num || static_cast<int>(space->num) != dg_selection_space()) {
        char b[160];
        std::snprintf(b, sizeof b, "made for kernel selection space %d, this build is %d (the kernels changed): run the sweep again",
                      space->kind == JVal::Num ? static_cast<int>(space->num) : -1, dg_selection_space());
        reason = b;
        return DG_ERR_TABLE_REFUSED;
    }
    const JVal* a = id->get("arch");
    if (!a || a->kind != JVal::Str || a->str != arch) {
        reason = "made for architecture " + (a && a->kind == JVal::Str ? a->str : std::string("?")) +
                 ", this device is " + arch;
        return DG_ERR_TABLE_REFUSED;
    }
    const JVal* d = id->get("driver");
    const JVal* r = id->get("runtime");
    if (!d || d->kind != JVal::Num || !r || r->kind != JVal::Num || static_cast<int>(d->num) != drv ||
        static_cast<int>(r->num) != rt) {
        char b[200];
        std::snprintf(b, sizeof b, "made with driver %d / runtime %d, this process has driver %d / runtime %d: tune and run with the same libraries",
                      d && d->kind == JVal::Num ? static_cast<int>(d->num) : -1,
                      r && r->kind == JVal::Num ? static_cast<int>(r->num) : -1, drv, rt);
        reason = b;
        return DG_ERR_TABLE_REFUSED;
    }
    const JVal* bid = id->get("build");
    if (!bid || bid->kind != JVal::Str || bid->str != build_id()) {
        reason = "made by library build " + (bid && bid->kind == JVal::Str ? bid->str : std::string("?")) +
                 ", this is " + build_id() + ": run the sweep again";
        return DG_ERR_TABLE_REFUSED;
    }
    if (const char* k = force_knob()) {
        reason = std::string("DG_FORCE_VARIANT=") + k +
                 " reroutes the decode dispatch away from what the table measured";
        return DG_ERR_TABLE_REFUSED;
    }
    const JVal* ents = root.get("entries");
    if (!ents || ents->kind != JVal::Arr) {
        reason = "table has no entries list";
        return DG_ERR_TABLE_REFUSED;
    }
    std::map<Key, Entry> tab;
    for (size_t i = 0; i < ents->arr.size(); ++i) {
        const JVal& e = ents->arr[i];
        const JVal* op = e.get("op");
        const JVal* M = e.get("M");
        const JVal* N = e.get("N");
        const JVal* K = e.get("K");
        char b[96];
        std::snprintf(b, sizeof b, "entry %zu: ", i);
        if (!op || op->kind != JVal::Str || !M || M->kind != JVal::Num || !N || N->kind != JVal::Num ||
            !K || K->kind != JVal::Num) {
            reason = std::string(b) + "missing op/M/N/K";
            return DG_ERR_TABLE_REFUSED;
        }
        const int opi = op_from_name(op->str);
        const int m = static_cast<int>(M->num);
        if (opi < 0) {
            reason = std::string(b) + "unknown op " + op->str;
            return DG_ERR_TABLE_REFUSED;
        }
        if (!valid_bucket(m)) {
            reason = std::string(b) + "rows " + std::to_string(m) + " are not a decode bucket";
            return DG_ERR_TABLE_REFUSED;
        }
        Entry en{};
        if (!parse_choice(e.get("pick"), en.choice)) {
            reason = std::string(b) + "missing or malformed pick";
            return DG_ERR_TABLE_REFUSED;
        }
        const std::string bad = check_choice(opi, en.choice);
        if (!bad.empty()) {
            reason = std::string(b) + bad;
            return DG_ERR_TABLE_REFUSED;
        }
        const JVal* us = e.get("pick_us");
        en.choice.from_table = 1;
        en.choice.table_us = (us && us->kind == JVal::Num) ? static_cast<float>(us->num) : 0.0f;
        tab[Key(opi, m, static_cast<int>(N->num), static_cast<int>(K->num))] = en;
    }
    if (out) *out = std::move(tab);
    return DG_OK;
}

}  // namespace

int bucket_rows(int M)
{
    static const int rows[] = {DG_ROWS_BUCKETS(DG_ROWS_AS_LIST)};
    for (int r : rows)
        if (r >= M) return r;
    return -1;
}

const char* op_key_name(int op) { return op_name(op); }

namespace {

std::atomic<int> g_numerics{DG_NUMERICS_FASTEST};

// The one family every bucket of `op` takes in the batch-invariant mode: the
// tensor cores, except for an fp8 head too wide for their shared-memory split
// activations, which stays on the CUDA cores at every row count.
bool cuda_core_family(int variant) { return variant == DG_VAR_CC_WARP || variant == DG_VAR_CC_BULK; }

int invariant_variant(int op, int K)
{
    if (op == DG_OP_HEAD_FP8_ARGMAX && K > kTcHeadMaxK) return DG_VAR_CC_WARP;
    return DG_VAR_TC;
}

bool same_family(int a, int b) { return a == b || (cuda_core_family(a) && cuda_core_family(b)); }

// The tensor-core linears cut K by a rule that depends on the row count beyond 128
// rows; params[1] = 1 fixes it to the shape alone.
void fix_split(int op, dg_choice* c)
{
    if (c->variant == DG_VAR_TC && (op == DG_OP_GEMV_BF16 || op == DG_OP_GATE_UP_SILU)) c->params[1] = 1;
}

}  // namespace

}  // namespace dg

using namespace dg;

extern "C" {

int dg_selection_space(void) { return 11; }

const char* dg_build_id(void) { return build_id(); }

dg_status dg_table_check(const char* path, const char* arch, int driver_version, int runtime_version,
                         int* entries, char* reason, size_t reason_cap)
{
    std::map<Key, Entry> tab;
    std::string why;
    dg_status s = load_impl(path, arch ? arch : "", driver_version, runtime_version, &tab, why);
    if (entries) *entries = (s == DG_OK) ? static_cast<int>(tab.size()) : 0;
    if (reason && reason_cap) std::snprintf(reason, reason_cap, "%s", why.c_str());
    return s;
}

dg_status dg_table_load(const char* path)
{
    dg_status s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    char arch[32];
    std::snprintf(arch, sizeof arch, "sm_%d%d", dev->cc_major, dev->cc_minor);
    std::map<Key, Entry> tab;
    std::string why;
    s = load_impl(path, arch, dev->driver_version, dev->runtime_version, &tab, why);
    if (s != DG_OK) {
        std::fprintf(stderr, "libdecodegemm: shape table %s refused: %s; defaults stay in effect\n",
                     path ? path : "(null)", why.c_str());
        return s;
    }
    std::lock_guard<std::mutex> lk(g_tmu);
    g_table = std::move(tab);
    g_table_path = path;
    if (std::getenv("DG_LOG"))
        std::fprintf(stderr, "libdecodegemm: %zu shapes from %s (%s, driver %d, runtime %d)\n",
                     g_table.size(), path, arch, dev->driver_version, dev->runtime_version);
    return DG_OK;
}

void dg_table_clear(void)
{
    std::lock_guard<std::mutex> lk(g_tmu);
    g_table.clear();
    g_table_path.clear();
}

int dg_table_entries(void)
{
    std::lock_guard<std::mutex> lk(g_tmu);
    return static_cast<int>(g_table.size());
}

dg_status dg_select(dg_op op, int M, int N, int K, dg_choice* out)
{
    if (!out || op < 0 || op >= DG_OP_COUNT) return DG_ERR_INVALID_ARG;
    const int b = bucket_rows(M);
    if (b < 0 || N < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (const char* k = force_knob()) {
        // DG_FORCE_VARIANT=variant:p0,p1,p2,p3 forces one kernel for every call.
        dg_choice c{};
        int v = 0, p[4] = {0, 0, 0, 0};
        if (std::sscanf(k, "%d:%d,%d,%d,%d", &v, &p[0], &p[1], &p[2], &p[3]) >= 1) {
            c.variant = v;
            for (int i = 0; i < 4; ++i) c.params[i] = p[i];
            if (check_choice(op, c).empty()) {
                *out = c;
                return DG_OK;
            }
        }
        return DG_ERR_BAD_VARIANT;
    }
    const bool invariant = g_numerics.load(std::memory_order_relaxed) == DG_NUMERICS_BATCH_INVARIANT;
    const int fam = invariant_variant(op, K);
    {
        std::lock_guard<std::mutex> lk(g_tmu);
        auto it = g_table.find(Key(op, b, N, K));
        if (it != g_table.end() && (!invariant || same_family(it->second.choice.variant, fam))) {
            *out = it->second.choice;
            if (invariant) fix_split(op, out);
            return DG_OK;
        }
    }
    default_choice(op, b, N, K, out);
    if (invariant && !same_family(out->variant, fam)) {
        // the family's own defaults: TC params are all derived from the shape, and a
        // CUDA-core head bucket is never out of its family here
        std::memset(out, 0, sizeof *out);
        out->variant = fam;
    }
    if (invariant) fix_split(op, out);
    return DG_OK;
}

dg_status dg_set_numerics(int mode)
{
    if (mode != DG_NUMERICS_FASTEST && mode != DG_NUMERICS_BATCH_INVARIANT) return DG_ERR_INVALID_ARG;
    g_numerics.store(mode);
    return DG_OK;
}

int dg_numerics(void) { return g_numerics.load(); }

}  // extern "C"
