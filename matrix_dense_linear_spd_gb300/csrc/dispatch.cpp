// C ABI of libbl.so: argument validation, flat kernel selection and launch.
//
// Selection follows BatchLAS "Flat kernel selection" (design page, sections 2 and 5):
//   * a choice is one spelling, "family[:field=value]...", used by tables, pins and traces;
//   * can_run is correctness only (the shape fits the variant), never speed (rule R3);
//   * speed lives only in the per-device tables: the nearest row's first runnable candidate
//     wins (rule R4; exact keys must match, dropping the rightmost exact key when none does;
//     distance sum w*|log2(row/key)|; ties to the row with the smaller keys);
//   * a pin (environment variable or bl_set_route) that does not parse or cannot run the shape
//     is an argument error (rule R6);
//   * BL_TRACE=1 prints one line per call.
#include "../../include/bl.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <map>
#include <mutex>
#include <sstream>
#include <string>
#include <tuple>
#include <vector>

#include "registry.h"

#include "_tuned_tables.inc"  // kTunedTables[]: {name, text}, generated from tuned/*.txt

namespace {

using bl::KernelEntry;

constexpr int64_t kMaxN = int64_t(1) << 20;
constexpr int64_t kMaxBatch = (int64_t(1) << 31) - 1;

thread_local std::string t_error;
thread_local std::string t_choice;
thread_local std::map<std::string, std::string> t_pins;  // op -> spelling ("" = none)

bl_status fail(bl_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return st;
}

const char *dtype_name(int d) {
    static const char *names[] = {"f32", "f64", "c64", "c128"};
    return (d >= 0 && d < 4) ? names[d] : "?";
}

std::string spelling(const KernelEntry &e);

// The compiled variants of a dtype with their spellings, built once.
struct Candidates {
    std::vector<const KernelEntry *> e;
    std::vector<std::string> sp;
};

const Candidates &candidates(int dtype) {
    static std::once_flag once;
    static Candidates all[4];
    std::call_once(once, [] {
        for (int d = 0; d < 4; ++d) {
            int count = 0;
            const KernelEntry *e = nullptr;
            switch (d) {
                case BL_F32: e = bl::entries_f32(&count); break;
                case BL_F64: e = bl::entries_f64(&count); break;
                case BL_C64: e = bl::entries_c64(&count); break;
                default: e = bl::entries_c128(&count); break;
            }
            for (int i = 0; i < count; ++i) {
                all[d].e.push_back(e + i);
                all[d].sp.push_back(spelling(e[i]));
            }
        }
    });
    static const Candidates none;
    return (dtype >= 0 && dtype < 4) ? all[dtype] : none;
}

std::string spelling(const KernelEntry &e) {
    char buf[64];
    if (e.family == 0) snprintf(buf, sizeof buf, "tile:p=%d:s=%d", e.p, e.s);
    else if (e.family == 2)   // nb bit 0: whole squares, bit 1: packed f32x2 update
        snprintf(buf, sizeof buf, "warp:p=%d:r=%d%s%s%s%s", e.p, e.s, (e.nb & 1) ? ":full=1" : "", (e.nb & 2) ? ":x2=1" : "",
                 (e.nb & 4) ? ":la=1" : "", (e.nb & 8) ? ":v2=1" : "");   // bit 2: look-ahead pivots, bit 3: float2-pair rows
    else if (e.family == 3)   // p: lanes per matrix; e: fully unrolled at n = NMAX
        snprintf(buf, sizeof buf, "thread:n=%d%s%s", e.nb, e.p == 2 ? ":p=2" : "", e.s == 1 ? ":e=1" : "");
    else if (e.s) snprintf(buf, sizeof buf, "blocked:nb=%d:tc=%d", e.nb, e.s);   // 2: the column-block tensor-core kernel
    else snprintf(buf, sizeof buf, "blocked:nb=%d", e.nb);
    return buf;
}

// Canonicalise a spelling: lower case, trimmed. "tile:4:8" is accepted as "tile:p=4:s=8".
std::string canon(std::string s) {
    auto issp = [](char c) { return c == ' ' || c == '\t' || c == '\n' || c == '\r'; };
    while (!s.empty() && issp(s.back())) s.pop_back();
    size_t b = 0;
    while (b < s.size() && issp(s[b])) ++b;
    s = s.substr(b);
    for (auto &c : s) c = static_cast<char>(tolower(static_cast<unsigned char>(c)));
    std::vector<std::string> parts;
    std::stringstream ss(s);
    std::string tok;
    while (std::getline(ss, tok, ':')) parts.push_back(tok);
    if (parts.empty()) return s;
    static const std::map<std::string, std::vector<std::string>> fields = {
        {"tile", {"p", "s"}}, {"warp", {"p", "r", "full", "x2", "la", "v2"}}, {"blocked", {"nb", "tc"}}, {"thread", {"n", "p", "e"}}};
    auto it = fields.find(parts[0]);
    if (it == fields.end()) return s;
    std::string out = parts[0];
    for (size_t i = 1; i < parts.size(); ++i) {
        std::string f = parts[i];
        if (f.find('=') == std::string::npos && i - 1 < it->second.size()) f = it->second[i - 1] + "=" + f;
        out += ":" + f;
    }
    return out;
}

enum Op { OP_POTRF = 0, OP_POSV = 1, OP_POTRS = 2 };
const char *op_name(int op) { return op == OP_POTRF ? "potrf" : op == OP_POSV ? "posv" : "potrs"; }

struct DeviceFacts {
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
    std::string key;
};

bool device_facts(DeviceFacts &f) {
    static std::mutex mu;
    static std::map<int, DeviceFacts> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) { f = it->second; return true; }
    DeviceFacts d;
    int v = 0;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    d.smem_optin = static_cast<size_t>(v);
    d.key = "sm_" + std::to_string(d.cc_major * 10 + d.cc_minor);
    cache[dev] = d;
    f = d;
    return true;
}

// Right-hand sides one pass of `e` takes, and whether the variant can run the shape at all.
int rhs_per_pass(const KernelEntry &e, int op, int64_t nrhs) {
    if (op == OP_POTRF || e.rhs_max < 0) return 0;
    if (e.family == 1) return static_cast<int>(nrhs);
    return static_cast<int>(std::min<int64_t>(nrhs, e.rhs_max));
}

bool can_run(const KernelEntry &e, int op, int64_t n, int64_t nrhs, const DeviceFacts &dev) {
    if (e.smem > dev.smem_optin) return false;
    if (op != OP_POTRF && e.rhs_max < 0) return false;  // factor-only variant
    if (e.family == 1) return e.cap == 0 || n <= e.cap;   // blocked: any n, or up to its panel capacity
    if (e.family == 2 || e.family == 3) return n <= e.cap;  // right-hand sides do not take rows
    return n + rhs_per_pass(e, op, nrhs) <= e.cap;
}

// ------------------------------------------------------------------ tables

struct Row {
    std::map<std::string, std::string> exact;  // dtype, uplo
    std::map<std::string, double> logk;        // n, nrhs, batch
    std::vector<std::string> ranked;
};

struct Table {
    std::vector<std::string> exact_keys;               // in "# keys:" order
    std::vector<std::pair<std::string, double>> log_keys;
    std::vector<Row> rows;
    std::string tag;
};

bool parse_table(const std::string &text, Table &t) {
    std::stringstream in(text);
    std::string line;
    while (std::getline(in, line)) {
        if (line.rfind("# keys:", 0) == 0) {
            std::stringstream ks(line.substr(7));
            std::string k;
            while (ks >> k) {
                std::vector<std::string> f;
                std::stringstream fs(k);
                std::string x;
                while (std::getline(fs, x, ':')) f.push_back(x);
                if (f.size() >= 2 && f[1] == "exact") t.exact_keys.push_back(f[0]);
                else if (f.size() >= 2 && f[1] == "log") t.log_keys.push_back({f[0], f.size() >= 3 ? atof(f[2].c_str()) : 1.0});
            }
            continue;
        }
        if (line.empty() || line[0] == '#') continue;
        size_t hash = line.find('#');
        if (hash != std::string::npos) line = line.substr(0, hash);
        std::vector<std::string> cells;
        std::stringstream cs(line);
        std::string c;
        while (std::getline(cs, c, '|')) cells.push_back(c);
        if (cells.size() < 2) continue;
        Row r;
        std::stringstream kv(cells[0]);
        std::string pair;
        while (kv >> pair) {
            size_t eq = pair.find('=');
            if (eq == std::string::npos) return false;
            std::string k = pair.substr(0, eq), v = pair.substr(eq + 1);
            bool is_exact = std::find(t.exact_keys.begin(), t.exact_keys.end(), k) != t.exact_keys.end();
            if (is_exact) r.exact[k] = v;
            else r.logk[k] = atof(v.c_str());
        }
        for (size_t i = 1; i < cells.size(); ++i) {
            std::stringstream one(cells[i]);
            std::string sp;
            if (one >> sp) r.ranked.push_back(canon(sp));
        }
        t.rows.push_back(r);
    }
    return true;
}

const Table *get_table(const std::string &op, const std::string &devkey, std::string &tag) {
    static std::mutex mu;
    static std::map<std::string, Table> cache;
    std::lock_guard<std::mutex> lk(mu);
    const std::string name = op + "." + devkey;
    auto it = cache.find(name);
    if (it != cache.end()) { tag = it->second.tag; return it->second.rows.empty() ? nullptr : &it->second; }
    Table t;
    std::string text;
    const char *dir = getenv("BL_TUNED_DIR");
    if (dir && *dir) {
        std::ifstream f(std::string(dir) + "/" + name + ".txt");
        if (f) { std::stringstream ss; ss << f.rdbuf(); text = ss.str(); t.tag = "override " + devkey; }
    }
    if (text.empty()) {
        // exact device first, then any table of the same op (nearest arch borrowing is not needed
        // for a single target; the tag records a borrow)
        for (const auto &kv : kTunedTables)
            if (name == kv[0]) { text = kv[1]; t.tag = devkey; }
        if (text.empty())
            for (const auto &kv : kTunedTables)
                if (std::string(kv[0]).rfind(op + ".", 0) == 0) { text = kv[1]; t.tag = std::string("borrowed ") + kv[0]; }
    }
    if (!text.empty() && !parse_table(text, t)) t.rows.clear();
    tag = t.tag;
    cache[name] = t;
    return cache[name].rows.empty() ? nullptr : &cache[name];
}

const Row *nearest_row(const Table &t, const std::map<std::string, std::string> &ex,
                       const std::map<std::string, double> &lg) {
    // all exact keys, then all but the rightmost one (tables are per dtype in effect: the
    // leading exact key is never dropped)
    const size_t nk = t.exact_keys.size();
    for (size_t keep = nk; keep + 1 >= nk && keep >= 1; --keep) {
        const Row *best = nullptr;
        double bestd = 0;
        for (const Row &r : t.rows) {
            bool match = true;
            for (size_t i = 0; i < keep; ++i) {
                const std::string &k = t.exact_keys[i];
                auto a = r.exact.find(k);
                auto b = ex.find(k);
                if (a == r.exact.end() || b == ex.end() || a->second != b->second) { match = false; break; }
            }
            if (!match) continue;
            double d = 0;
            for (const auto &kw : t.log_keys) {
                auto a = r.logk.find(kw.first);
                auto b = lg.find(kw.first);
                if (a == r.logk.end() || b == lg.end() || a->second <= 0 || b->second <= 0) continue;
                d += kw.second * std::fabs(std::log2(a->second / b->second));
            }
            bool better = !best || d < bestd - 1e-9;
            if (!better && best && std::fabs(d - bestd) <= 1e-9) {
                for (const auto &kw : t.log_keys) {  // tie: the smaller keys win
                    double x = r.logk.count(kw.first) ? r.logk.at(kw.first) : 0;
                    double y = best->logk.count(kw.first) ? best->logk.at(kw.first) : 0;
                    if (x != y) { better = x < y; break; }
                }
            }
            if (better) { best = &r; bestd = d; }
        }
        if (best) return best;
    }
    return nullptr;
}

// ------------------------------------------------------------------ choice

struct Choice {
    const KernelEntry *e = nullptr;
    std::string how;  // "pin", "table <tag> row ...", "last resort"
};

std::string env_pin(int op) {
    static std::once_flag once;
    static std::string pins[3];
    std::call_once(once, [] {
        const char *names[3] = {"BL_POTRF_ROUTE", "BL_POSV_ROUTE", "BL_POTRS_ROUTE"};
        for (int i = 0; i < 3; ++i) {
            const char *v = getenv(names[i]);
            pins[i] = v ? v : "";
        }
    });
    return pins[op];
}

bl_status choose_on(const DeviceFacts &dev, int op, int dtype, int uplo, int64_t n, int64_t nrhs,
                    int64_t batch, Choice &out) {
    const Candidates &cs = candidates(dtype);
    const auto &cands = cs.e;
    std::string pin;
    auto tp = t_pins.find(op_name(op));
    if (tp != t_pins.end() && !tp->second.empty()) pin = tp->second;
    else pin = env_pin(op);
    std::string cp = canon(pin);
    if (!cp.empty() && cp != "auto") {
        for (size_t i = 0; i < cands.size(); ++i)
            if (cs.sp[i] == cp) {
                const KernelEntry *e = cands[i];
                if (!can_run(*e, op, n, nrhs, dev))
                    return fail(BL_ERR_INVALID_ARGUMENT, "%s route pin '%s' cannot run %s n=%lld nrhs=%lld",
                                op_name(op), pin.c_str(), dtype_name(dtype), (long long)n, (long long)nrhs);
                out.e = e;
                out.how = "pin";
                return BL_SUCCESS;
            }
        return fail(BL_ERR_INVALID_ARGUMENT, "%s route pin '%s' names no %s kernel", op_name(op), pin.c_str(),
                    dtype_name(dtype));
    }
    std::string tag;
    const Table *t = get_table(op == OP_POTRS ? "posv" : op_name(op), dev.key, tag);
    if (t) {
        std::map<std::string, std::string> ex = {{"dtype", dtype_name(dtype)}, {"uplo", uplo ? "U" : "L"}};
        std::map<std::string, double> lg = {{"n", double(n)}, {"batch", double(batch)}};
        if (op != OP_POTRF) lg["nrhs"] = double(nrhs);
        if (const Row *r = nearest_row(*t, ex, lg)) {
            for (const std::string &sp : r->ranked)
                for (size_t i = 0; i < cands.size(); ++i)
                    if (cs.sp[i] == sp && can_run(*cands[i], op, n, nrhs, dev)) {
                        const KernelEntry *e = cands[i];
                        char buf[160];
                        snprintf(buf, sizeof buf, "table %s row n=%g batch=%g", tag.c_str(),
                                 r->logk.count("n") ? r->logk.at("n") : 0.0,
                                 r->logk.count("batch") ? r->logk.at("batch") : 0.0);
                        out.e = e;
                        out.how = buf;
                        return BL_SUCCESS;
                    }
        }
    }
    // last resort: the smallest register-resident variant (warp or tile) that holds the shape,
    // preferring the warp family on a tie, else the blocked family
    const KernelEntry *best = nullptr;
    for (const KernelEntry *e : cands) {
        if (e->family == 1 || !can_run(*e, op, n, nrhs, dev)) continue;
        if (!best || e->cap < best->cap || (e->cap == best->cap && e->family > best->family) ||
            (e->cap == best->cap && e->family == best->family && e->p > best->p))
            best = e;
    }
    if (!best)
        for (const KernelEntry *e : cands)
            if (e->family == 1 && can_run(*e, op, n, nrhs, dev)) { best = e; break; }
    if (!best) return fail(BL_ERR_NO_ROUTE, "no kernel can run %s %s n=%lld", op_name(op), dtype_name(dtype), (long long)n);
    out.e = best;
    out.how = "last resort";
    return BL_SUCCESS;
}

// Resolved choices, per thread, keyed by everything the choice depends on (device, op, dtype,
// uplo, n, nrhs, batch and the pin in force): a repeated call skips the table search.
struct ChoiceKey {
    int dev, op, dtype, uplo;
    int64_t n, nrhs, batch;
    std::string pin;
    bool operator<(const ChoiceKey &o) const {
        return std::tie(dev, op, dtype, uplo, n, nrhs, batch, pin) <
               std::tie(o.dev, o.op, o.dtype, o.uplo, o.n, o.nrhs, o.batch, o.pin);
    }
};
thread_local std::map<ChoiceKey, Choice> t_choice_cache;

bl_status choose(int op, int dtype, int uplo, int64_t n, int64_t nrhs, int64_t batch, Choice &out) {
    int devno = 0;
    if (cudaGetDevice(&devno) != cudaSuccess) return fail(BL_ERR_CUDA, "cannot query the current CUDA device");
    auto tp = t_pins.find(op_name(op));
    ChoiceKey key{devno, op, dtype, uplo, n, op == OP_POTRF ? 0 : nrhs, batch,
                  (tp != t_pins.end() && !tp->second.empty()) ? tp->second : env_pin(op)};
    auto hit = t_choice_cache.find(key);
    if (hit != t_choice_cache.end()) {
        out = hit->second;
        return BL_SUCCESS;
    }
    DeviceFacts dev;
    if (!device_facts(dev)) return fail(BL_ERR_CUDA, "cannot query the current CUDA device");
    bl_status st = choose_on(dev, op, dtype, uplo, n, nrhs, batch, out);
    if (st == BL_SUCCESS) {
        if (t_choice_cache.size() > 4096) t_choice_cache.clear();
        t_choice_cache[key] = out;
    }
    return st;
}

bool trace_on() {
    static int on = -1;
    if (on < 0) {
        const char *v = getenv("BL_TRACE");
        on = (v && *v && strcmp(v, "0") != 0) ? 1 : 0;
    }
    return on == 1;
}

size_t elem_size(int dtype) {
    switch (dtype) {
        case BL_F32: return 4;
        case BL_F64: return 8;
        case BL_C64: return 8;
        case BL_C128: return 16;
        default: return 0;
    }
}

bl_status validate(int op, int uplo, int dtype, int64_t n, int64_t nrhs, int64_t batch, const void *A,
                   int64_t lda, int64_t stride_a, const void *B, int64_t ldb, int64_t stride_b,
                   const int32_t *info) {
    if (uplo != BL_LOWER && uplo != BL_UPPER) return fail(BL_ERR_INVALID_ARGUMENT, "uplo %d is not BL_LOWER/BL_UPPER", uplo);
    if (dtype < BL_F32 || dtype > BL_C128) return fail(BL_ERR_INVALID_ARGUMENT, "unknown dtype %d", dtype);
    if (n < 1 || n > kMaxN) return fail(BL_ERR_INVALID_ARGUMENT, "n=%lld outside [1, %lld]", (long long)n, (long long)kMaxN);
    if (batch < 1 || batch > kMaxBatch)
        return fail(BL_ERR_INVALID_ARGUMENT, "batch=%lld outside [1, %lld]", (long long)batch, (long long)kMaxBatch);
    if (A == nullptr) return fail(BL_ERR_INVALID_ARGUMENT, "A is NULL");
    const size_t es = elem_size(dtype);
    if (reinterpret_cast<uintptr_t>(A) % es != 0)
        return fail(BL_ERR_INVALID_ARGUMENT, "A is not aligned to its %zu-byte element", es);
    if (info != nullptr && reinterpret_cast<uintptr_t>(info) % 4 != 0)
        return fail(BL_ERR_INVALID_ARGUMENT, "info is not 4-byte aligned");
    if (lda < n) return fail(BL_ERR_INVALID_ARGUMENT, "lda=%lld < n=%lld", (long long)lda, (long long)n);
    if (lda > INT64_MAX / n / 16) return fail(BL_ERR_INVALID_ARGUMENT, "lda=%lld too large", (long long)lda);
    if (stride_a < lda * n)
        return fail(BL_ERR_INVALID_ARGUMENT, "stride_a=%lld < lda*n=%lld (items overlap)", (long long)stride_a, (long long)(lda * n));
    if (stride_a > INT64_MAX / batch / 16) return fail(BL_ERR_INVALID_ARGUMENT, "stride_a=%lld too large", (long long)stride_a);
    if (op != OP_POTRS && info == nullptr) return fail(BL_ERR_INVALID_ARGUMENT, "info is NULL");
    if (op != OP_POTRF) {
        if (nrhs < 1 || nrhs > kMaxN) return fail(BL_ERR_INVALID_ARGUMENT, "nrhs=%lld outside [1, %lld]", (long long)nrhs, (long long)kMaxN);
        if (B == nullptr) return fail(BL_ERR_INVALID_ARGUMENT, "B is NULL");
        if (reinterpret_cast<uintptr_t>(B) % es != 0)
            return fail(BL_ERR_INVALID_ARGUMENT, "B is not aligned to its %zu-byte element", es);
        if (ldb < n) return fail(BL_ERR_INVALID_ARGUMENT, "ldb=%lld < n=%lld", (long long)ldb, (long long)n);
        if (ldb > INT64_MAX / nrhs / 16) return fail(BL_ERR_INVALID_ARGUMENT, "ldb=%lld too large", (long long)ldb);
        if (stride_b < ldb * nrhs)
            return fail(BL_ERR_INVALID_ARGUMENT, "stride_b=%lld < ldb*nrhs=%lld (items overlap)", (long long)stride_b, (long long)(ldb * nrhs));
        if (stride_b > INT64_MAX / batch / 16) return fail(BL_ERR_INVALID_ARGUMENT, "stride_b=%lld too large", (long long)stride_b);
    }
    return BL_SUCCESS;
}

bl_status run(int op, int uplo, int dtype, int64_t n, int64_t nrhs, int64_t batch, void *A, int64_t lda,
              int64_t stride_a, void *B, int64_t ldb, int64_t stride_b, int32_t *info, bl_stream_t stream) {
    t_error.clear();
    bl_status st = validate(op, uplo, dtype, n, nrhs, batch, A, lda, stride_a, B, ldb, stride_b, info);
    if (st != BL_SUCCESS) return st;
    Choice ch;
    st = choose(op, dtype, uplo, n, nrhs, batch, ch);
    if (st != BL_SUCCESS) return st;
    t_choice = spelling(*ch.e);
    if (trace_on())
        fprintf(stderr, "bl: %s %s uplo=%c n=%lld nrhs=%lld batch=%lld -> %s [%s]\n", op_name(op), dtype_name(dtype),
                uplo ? 'U' : 'L', (long long)n, (long long)(op == OP_POTRF ? 0 : nrhs), (long long)batch,
                t_choice.c_str(), ch.how.c_str());
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t es = elem_size(dtype);
    bl::BatchArgs a{};
    a.n = static_cast<int>(n);
    a.upper = uplo;
    a.batch = batch;
    a.A = A;
    a.lda = lda;
    a.stride_a = stride_a;
    a.ldb = ldb;
    a.stride_b = stride_b;
    a.info = info;
    int64_t done = 0;
    do {
        const int pass = rhs_per_pass(*ch.e, op, nrhs - done);
        if (op == OP_POTRF) a.mode = bl::MODE_POTRF;
        else if (op == OP_POSV && done == 0) a.mode = bl::MODE_POSV;
        else a.mode = bl::MODE_POTRS;  // later passes of posv read info and skip failed items
        a.nrhs = pass;
        a.B = (op == OP_POTRF) ? nullptr : static_cast<char *>(B) + static_cast<size_t>(done * ldb) * es;
        cudaError_t e = ch.e->launch(a, s);
        if (e != cudaSuccess) return fail(BL_ERR_CUDA, "%s launch failed: %s", t_choice.c_str(), cudaGetErrorString(e));
        done += pass;
    } while (op != OP_POTRF && done < nrhs);
    return BL_SUCCESS;
}

}  // namespace

extern "C" {

bl_status bl_potrf(bl_uplo uplo, bl_dtype dtype, int64_t n, int64_t batch, void *A, int64_t lda,
                   int64_t stride_a, int32_t *info, bl_stream_t stream) {
    return run(OP_POTRF, uplo, dtype, n, 0, batch, A, lda, stride_a, nullptr, 0, 0, info, stream);
}

bl_status bl_posv(bl_uplo uplo, bl_dtype dtype, int64_t n, int64_t nrhs, int64_t batch, void *A, int64_t lda,
                  int64_t stride_a, void *B, int64_t ldb, int64_t stride_b, int32_t *info, bl_stream_t stream) {
    return run(OP_POSV, uplo, dtype, n, nrhs, batch, A, lda, stride_a, B, ldb, stride_b, info, stream);
}

bl_status bl_potrs(bl_uplo uplo, bl_dtype dtype, int64_t n, int64_t nrhs, int64_t batch, const void *A,
                   int64_t lda, int64_t stride_a, void *B, int64_t ldb, int64_t stride_b, bl_stream_t stream) {
    return run(OP_POTRS, uplo, dtype, n, nrhs, batch, const_cast<void *>(A), lda, stride_a, B, ldb, stride_b,
               nullptr, stream);
}

const char *bl_status_string(bl_status s) {
    switch (s) {
        case BL_SUCCESS: return "success";
        case BL_ERR_INVALID_ARGUMENT: return "invalid argument";
        case BL_ERR_NO_ROUTE: return "no kernel can run the shape";
        case BL_ERR_CUDA: return "CUDA error";
        case BL_ERR_INTERNAL: return "internal error";
        default: return "unknown status";
    }
}

const char *bl_last_error(void) { return t_error.c_str(); }
const char *bl_last_choice(void) { return t_choice.c_str(); }
int bl_version(void) { return 100; }

// Thread-local route pin, overriding BL_<OP>_ROUTE for this thread. op is "potrf", "posv" or
// "potrs"; spelling NULL or "" clears the pin, "auto" selects by table. Returns BL_SUCCESS, or
// BL_ERR_INVALID_ARGUMENT for an unknown op. The spelling itself is checked at the next call.
bl_status bl_set_route(const char *op, const char *spelling_) {
    if (!op || (strcmp(op, "potrf") && strcmp(op, "posv") && strcmp(op, "potrs")))
        return fail(BL_ERR_INVALID_ARGUMENT, "unknown op for a route pin");
    t_pins[op] = spelling_ ? spelling_ : "";
    return BL_SUCCESS;
}

// Host-only selection for a synthetic device (no CUDA call): op 0/1/2 = potrf/posv/potrs.
// Returns "<spelling> [<how>]" or "error: <message>". For tests of the selection layer.
const char *bl_select_debug(int op, bl_dtype dtype, bl_uplo uplo, int64_t n, int64_t nrhs, int64_t batch,
                            const char *devkey, int64_t smem_optin) {
    static thread_local std::string s;
    DeviceFacts dev;
    dev.key = devkey ? devkey : "sm_103";
    dev.smem_optin = static_cast<size_t>(smem_optin);
    Choice ch;
    bl_status st = validate(op, uplo, dtype, n, op == OP_POTRF ? 0 : nrhs, batch, reinterpret_cast<void *>(16), n,
                            n * n, reinterpret_cast<void *>(16), n, n * std::max<int64_t>(nrhs, 1),
                            reinterpret_cast<int32_t *>(16));
    if (st == BL_SUCCESS) st = choose_on(dev, op, dtype, uplo, n, nrhs, batch, ch);
    s = (st == BL_SUCCESS) ? spelling(*ch.e) + " [" + ch.how + "]" : "error: " + t_error;
    return s.c_str();
}

// Number of compiled kernel variants for a dtype, and the spelling of variant i (for sweeps
// and tests). Returns NULL when i is out of range.
int bl_num_routes(bl_dtype dtype) { return static_cast<int>(candidates(dtype).e.size()); }

const char *bl_route_name(bl_dtype dtype, int i) {
    static thread_local std::string s;
    const auto &c = candidates(dtype);
    if (i < 0 || i >= static_cast<int>(c.e.size())) return nullptr;
    s = c.sp[i];
    return s.c_str();
}

// Capacity of variant i: the largest n + rhs-per-pass it holds (0 = any) and the right-hand
// sides it solves per pass (0 = any). Returns -1 when i is out of range.
int bl_route_capacity(bl_dtype dtype, int i, int *rhs_per_pass_out) {
    const auto &c = candidates(dtype);
    if (i < 0 || i >= static_cast<int>(c.e.size())) return -1;
    if (rhs_per_pass_out) *rhs_per_pass_out = c.e[i]->rhs_max;
    return c.e[i]->cap;
}

}  // extern "C"
