// Tracing and configuration logging of libpagedattn.so (host side).
//
// * Every C-ABI entry point opens an NVTX range named after itself, so a
//   timeline tool shows which call issued which kernels.  Without a tool
//   attached an NVTX call is a cheap no-op.
// * With the environment variable PAGEDATTN_LOG set (to anything but "0"),
//   the launch configuration each call chose -- kernel variant, grid, split
//   size -- is printed to stderr the first time it is used, one line per
//   distinct configuration, so the one path that runs is on record.
// * PAGEDATTN_DECODE_CHUNK=n (n >= 1) sets the smallest split-K chunk of the
//   decode kernels to n 16-key units instead of 16, so that small test
//   problems are split across many CTAs and exercise the log-sum-exp merge.
//   It changes only how the work is cut, never what is computed.
// * PAGEDATTN_PREFILL_WAIT_NS=n (n >= 1) sets the time limit of every wait
//   in the prefill kernel to n nanoseconds instead of 2 s.  A tiny limit makes
//   the waits run out, which is how the tests exercise the timeout path
//   (PA_ERR_TIMEOUT in the status word, a clean exit, a usable context).
// * PAGEDATTN_PREFILL_PATH=fused|separate picks how attn_prefill_varlen_causal
//   runs a call with prefill entries: one persistent kernel for the decode
//   rows and the prefill tiles (plus the merge of split decode rows), or the
//   split-K decode, the plan and the prefill as separate kernels.  Both compute
//   the same result; the tests run both.
// * PAGEDATTN_PREFILL_PAIR=1 runs the stand-alone prefill kernel as CTA pairs
//   (one M = 256 MMA per tile over two SMs; head_dim 128 only) instead of
//   single CTAs (the default, measured faster); the tests cover both.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <string>

namespace pa {

struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

inline bool log_enabled() {
    const char* v = std::getenv("PAGEDATTN_LOG");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
}

// Print a configuration line once per distinct text (when PAGEDATTN_LOG is set).
inline void log_config(const char* fmt, ...) {
    if (!log_enabled()) return;
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    static std::mutex mu;
    static std::set<std::string> seen;
    std::lock_guard<std::mutex> lk(mu);
    if (seen.insert(buf).second) std::fprintf(stderr, "[pagedattn] %s\n", buf);
}

// Smallest split-K chunk in units: PAGEDATTN_DECODE_CHUNK if set to an integer
// in [1, 1 << 20], else `dflt`.
inline int decode_min_chunk(int dflt) {
    const char* v = std::getenv("PAGEDATTN_DECODE_CHUNK");
    if (v == nullptr || v[0] == '\0') return dflt;
    char* end = nullptr;
    const long n = std::strtol(v, &end, 10);
    if (end == v || *end != '\0' || n < 1 || n > (1 << 20)) return dflt;
    return (int)n;
}

// Wait limit of the prefill kernel in ns: PAGEDATTN_PREFILL_WAIT_NS if set to an
// integer in [1, 60 s], else `dflt`.
inline unsigned long long prefill_wait_ns(unsigned long long dflt) {
    const char* v = std::getenv("PAGEDATTN_PREFILL_WAIT_NS");
    if (v == nullptr || v[0] == '\0') return dflt;
    char* end = nullptr;
    const long long n = std::strtoll(v, &end, 10);
    if (end == v || *end != '\0' || n < 1 || n > 60000000000ll) return dflt;
    return (unsigned long long)n;
}

// 1: CTA pairs, 2: single CTAs, 0: not set (the library's default).
inline int prefill_pair_override() {
    const char* v = std::getenv("PAGEDATTN_PREFILL_PAIR");
    if (v == nullptr) return 0;
    if (std::strcmp(v, "1") == 0) return 1;
    if (std::strcmp(v, "0") == 0) return 2;
    return 0;
}

// 1: one fused launch, 2: separate kernels, 0: not set (the library's default).
inline int prefill_path_override() {
    const char* v = std::getenv("PAGEDATTN_PREFILL_PATH");
    if (v == nullptr) return 0;
    if (std::strcmp(v, "fused") == 0) return 1;
    if (std::strcmp(v, "separate") == 0) return 2;
    return 0;
}

}  // namespace pa
