// Eager K/V writeback into pages ("Inside Ion", section "IonAttention in One
// Paragraph": KV pages are written back eagerly as they are produced).
//
// Each warp moves new rows (two at a time): it finds a row's sequence by counting
// the cu_seqlens_new entries at or below it (one coalesced load per 32 sequences),
// resolves (page, slot) through the block table, and
// copies the row's [Hkv][D] K and V vectors with 16-byte vector loads and
// stores.  A bit-exact copy; nothing else in the pools is written.
//
// kv_write_paged_rope fuses the step before it ("The Stack Below the Stack,
// Part 2", section 2.1: fused Q-norm, KV-RoPE and K-insert): each K head row
// (and, optionally, each query head row, in place) is RMS-normalised when a
// weight is given and rotated by the rotary position embedding at the row's
// position, in fp32, then rounded once to bf16; V rows are copied.  Lane l of
// the token's warp owns the pairs (i, i + D/2) for i in [l * D/64, (l+1) *
// D/64), so each pair is rotated by one thread and the cos / sin of the
// token's angles are computed once and reused for every head.  Angles are
// reduced exactly: the host passes frac(theta_i / 2 pi) as a 64-bit binary
// fraction, the position times it (mod 2^64) is the angle in turns, and
// sincospif turns its top 24 bits into cos and sin.
//
// kv_write_paged_fp8 is the writeback of an FP8 (e4m3) cache ("The Stack
// Below the Stack, Part 2", closing recipe: FP8 KV): element x of KV head g
// is stored as the e4m3 code nearest to x / scale[g] (fp32 quotient, round to
// nearest even, saturating at +-448).  K rows keep the [page][Hkv][slot][D]
// layout; V is transposed inside each page block, [page][Hkv][D][slot], so
// that the decode kernel reads the keys of one value column as one word.
#include "pa_common.cuh"
#include "pa_host.h"
#include "pa_trace.h"

#include <cmath>
#include <cuda_fp8.h>

namespace pa {
namespace kvw {

constexpr int kWarps = 8;

// Sequence of new row t: the last b with cu_new[b] <= t, which is the number of
// entries <= t minus one (cu_new is non-decreasing, so they form a prefix; the
// last of several equal entries is the non-empty sequence holding t).  The warp
// counts them 32 at a time with coalesced loads: one memory round trip for up to
// 31 sequences, instead of a chain of dependent binary-search loads.
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu_new, int batch, int t) {
    const int lane = threadIdx.x & 31;
    int cnt = 0;
    for (int c = 0; c <= batch; c += 32) {
        const int idx = c + lane;
        const int v = idx <= batch ? __ldg(cu_new + idx) : 0x7fffffff;
        cnt += __popc(__ballot_sync(0xffffffffu, v <= t));
    }
    return cnt - 1;
}

// Sequences of new rows t0 and t1 (see find_seq), counted in one pass.
__device__ __forceinline__ void find_seq2(const int32_t* __restrict__ cu_new, int batch, int t0, int t1, int& b0,
                                          int& b1) {
    const int lane = threadIdx.x & 31;
    int c0 = 0, c1 = 0;
    for (int c = 0; c <= batch; c += 32) {
        const int idx = c + lane;
        const int v = idx <= batch ? __ldg(cu_new + idx) : 0x7fffffff;
        c0 += __popc(__ballot_sync(0xffffffffu, v <= t0));
        c1 += __popc(__ballot_sync(0xffffffffu, v <= t1));
    }
    b0 = c0 - 1;
    b1 = c1 - 1;
}

// One warp moves two new rows at a time (rows t and t + stride of its grid-stride walk):
// both rows' vectors are loaded first, then both rows' (sequence, page, slot) lookups run
// side by side -- each is a chain of dependent loads (cu_seqlens, seq_lens, block table) --
// and both rows are stored.  Two independent chains per warp hide each other's latency.
__global__ void __launch_bounds__(kWarps * 32) kv_write_kernel(
    __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ v_pool, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, const int32_t* __restrict__ cu_new, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, int num_pages, int max_pages, int batch, int total_new, int page_size,
    int num_kv_heads, int head_dim, int32_t* status) {
    pdl_launch_dependents();  // the next kernel (e.g. the decode) may start; it waits for our writes
    const int lane = threadIdx.x & 31;
    const int vec_per_head = head_dim / 8;  // 16-byte vectors per row
    const int vec_per_tok = num_kv_heads * vec_per_head;
    const int nwarps = gridDim.x * kWarps;
    for (int ta = blockIdx.x * kWarps + (threadIdx.x >> 5); ta < total_new; ta += 2 * nwarps) {
        const int tt[2] = {ta, ta + nwarps};
        uint4 kr[2][2], vr[2][2];  // [row][vector lane, lane + 32]
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            kr[u][0] = kr[u][1] = vr[u][0] = vr[u][1] = make_uint4(0, 0, 0, 0);
            if (tt[u] < total_new) {
                const uint4* ks = reinterpret_cast<const uint4*>(k_new + (size_t)tt[u] * num_kv_heads * head_dim);
                const uint4* vs = reinterpret_cast<const uint4*>(v_new + (size_t)tt[u] * num_kv_heads * head_dim);
                if (lane < vec_per_tok) {
                    kr[u][0] = __ldg(ks + lane);
                    vr[u][0] = __ldg(vs + lane);
                }
                if (lane + 32 < vec_per_tok) {
                    kr[u][1] = __ldg(ks + lane + 32);
                    vr[u][1] = __ldg(vs + lane + 32);
                }
            }
        }
        int bb[2];
        find_seq2(cu_new, batch, tt[0], tt[1] < total_new ? tt[1] : tt[0], bb[0], bb[1]);
        int c0[2], n_b[2], L[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = min(max(bb[u], 0), batch - 1);  // (checked below)
            c0[u] = __ldg(cu_new + b);
            n_b[u] = __ldg(cu_new + b + 1) - c0[u];
            L[u] = __ldg(seq_lens + b);
        }
        int phys[2], slot[2];
        bool okk[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = bb[u];
            const int i = tt[u] - c0[u];
            const int pos = L[u] - n_b[u] + i;
            okk[u] = tt[u] < total_new;
            phys[u] = -1;
            slot[u] = 0;
            if (okk[u] && (b < 0 || b >= batch || n_b[u] <= 0 || i >= n_b[u] || pos < 0 ||
                           pos >= max_pages * page_size)) {
                if (lane == 0) report(status, PA_ERR_BAD_LEN);
                okk[u] = false;
            }
            if (okk[u]) {
                phys[u] = __ldg(block_table + (size_t)b * max_pages + pos / page_size);
                slot[u] = pos % page_size;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (!okk[u]) continue;
            if (phys[u] < 0 || phys[u] >= num_pages) {
                if (lane == 0) report(status, PA_ERR_BAD_PAGE);
                continue;
            }
            const uint4* ks = reinterpret_cast<const uint4*>(k_new + (size_t)tt[u] * num_kv_heads * head_dim);
            const uint4* vs = reinterpret_cast<const uint4*>(v_new + (size_t)tt[u] * num_kv_heads * head_dim);
            for (int v = lane; v < vec_per_tok; v += 32) {
                const int g = v / vec_per_head;
                const int c = v - g * vec_per_head;
                const size_t dst = (((size_t)phys[u] * num_kv_heads + g) * page_size + slot[u]) * head_dim / 8 + c;
                const uint4 kv = v == lane ? kr[u][0] : (v == lane + 32 ? kr[u][1] : __ldg(ks + v));
                const uint4 vv = v == lane ? vr[u][0] : (v == lane + 32 ? vr[u][1] : __ldg(vs + v));
                reinterpret_cast<uint4*>(k_pool)[dst] = kv;
                reinterpret_cast<uint4*>(v_pool)[dst] = vv;
            }
        }
    }
}

struct RopeParams {
    __nv_bfloat16* k_pool;
    __nv_bfloat16* v_pool;
    const __nv_bfloat16* k_new;
    const __nv_bfloat16* v_new;
    __nv_bfloat16* q;  // may be null
    const __nv_bfloat16* q_norm_w;  // may be null
    const __nv_bfloat16* k_norm_w;  // may be null
    const int32_t* cu_new;
    const int32_t* seq_lens;
    const int32_t* block_table;
    int32_t* status;
    int num_pages, max_pages, batch, total_new, page_size, Hkv, Hq;
    float eps;
    unsigned long long turns[64];  // frac(base^(-2i/D) / (2 pi)) * 2^64, i < D/2
};

// Pair elements of one head row held by a lane: x1[j] = row[i_j], x2[j] = row[i_j + D/2].
template <int D>
struct PairIO {
    static constexpr int PPL = D / 64;  // pairs per lane
    __device__ static void load(const __nv_bfloat16* row, int lane, float* x1, float* x2) {
        if constexpr (PPL == 2) {
            const __nv_bfloat162 a = reinterpret_cast<const __nv_bfloat162*>(row)[lane];
            const __nv_bfloat162 b = reinterpret_cast<const __nv_bfloat162*>(row + D / 2)[lane];
            x1[0] = __low2float(a);
            x1[1] = __high2float(a);
            x2[0] = __low2float(b);
            x2[1] = __high2float(b);
        } else {
            x1[0] = __bfloat162float(row[lane]);
            x2[0] = __bfloat162float(row[lane + D / 2]);
        }
    }
    __device__ static void store(__nv_bfloat16* row, int lane, const float* y1, const float* y2) {
        if constexpr (PPL == 2) {
            reinterpret_cast<__nv_bfloat162*>(row)[lane] = __floats2bfloat162_rn(y1[0], y1[1]);
            reinterpret_cast<__nv_bfloat162*>(row + D / 2)[lane] = __floats2bfloat162_rn(y2[0], y2[1]);
        } else {
            row[lane] = __float2bfloat16_rn(y1[0]);
            row[lane + D / 2] = __float2bfloat16_rn(y2[0]);
        }
    }
};

// Normalise (optional) and rotate NH head rows held as pairs.  All NH rows
// are loaded before any is processed, so NH loads are in flight at once.
template <int D, int NH>
__device__ __forceinline__ void rope_rows(const __nv_bfloat16* src, size_t src_stride, __nv_bfloat16* const* dst,
                                          const __nv_bfloat16* w, float eps, int lane, const float* c,
                                          const float* s) {
    constexpr int PPL = D / 64;
    float x1[NH][PPL], x2[NH][PPL];
#pragma unroll
    for (int h = 0; h < NH; ++h) PairIO<D>::load(src + h * src_stride, lane, x1[h], x2[h]);
    if (w != nullptr) {
        float w1[PPL], w2[PPL];
        PairIO<D>::load(w, lane, w1, w2);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < PPL; ++j) ss += x1[h][j] * x1[h][j] + x2[h][j] * x2[h][j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float r = rsqrtf(ss * (1.f / D) + eps);
#pragma unroll
            for (int j = 0; j < PPL; ++j) {
                x1[h][j] *= r * w1[j];
                x2[h][j] *= r * w2[j];
            }
        }
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        float y1[PPL], y2[PPL];
#pragma unroll
        for (int j = 0; j < PPL; ++j) {
            y1[j] = x1[h][j] * c[j] - x2[h][j] * s[j];
            y2[j] = x2[h][j] * c[j] + x1[h][j] * s[j];
        }
        PairIO<D>::store(dst[h], lane, y1, y2);
    }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) kv_write_rope_kernel(const __grid_constant__ RopeParams p) {
    constexpr int PPL = D / 64;
    pdl_launch_dependents();  // the next kernel (e.g. the decode) may start; it waits for our writes
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * kWarps;
    for (int t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < p.total_new; t += nwarps) {
        const int b = find_seq(p.cu_new, p.batch, t);
        if (b < 0 || b >= p.batch) {
            if (lane == 0) report(p.status, PA_ERR_BAD_LEN);
            continue;
        }
        const int n_b = __ldg(p.cu_new + b + 1) - __ldg(p.cu_new + b);
        const int i = t - __ldg(p.cu_new + b);
        const int L = __ldg(p.seq_lens + b);
        const int pos = L - n_b + i;
        if (n_b <= 0 || i >= n_b || pos < 0 || pos >= p.max_pages * p.page_size) {
            if (lane == 0) report(p.status, PA_ERR_BAD_LEN);
            continue;
        }
        // the page is looked up now and used after the query rows, which need only the position
        const int phys = __ldg(p.block_table + (size_t)b * p.max_pages + pos / p.page_size);
        const int slot = pos % p.page_size;
        // cos / sin of this position's angles, one pair at a time
        float c[PPL], s[PPL];
#pragma unroll
        for (int j = 0; j < PPL; ++j) {
            const unsigned long long turn = (unsigned long long)pos * p.turns[lane * PPL + j];  // mod 2^64
            const float frac = (float)(unsigned)(turn >> 40) * 0x1p-24f;                     // exact
            sincospif(2.f * frac, &s[j], &c[j]);
        }
        if (p.q != nullptr) {
            __nv_bfloat16* qrow = p.q + (size_t)t * p.Hq * D;
            // eight head rows per batch of loads: one warp keeps 2 KB in flight
            int h = 0;
            for (; h + 8 <= p.Hq; h += 8) {
                __nv_bfloat16* qd[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) qd[k] = qrow + (h + k) * D;
                rope_rows<D, 8>(qrow + h * D, D, qd, p.q_norm_w, p.eps, lane, c, s);
            }
            for (; h + 4 <= p.Hq; h += 4) {
                __nv_bfloat16* qd[4] = {qrow + h * D, qrow + (h + 1) * D, qrow + (h + 2) * D, qrow + (h + 3) * D};
                rope_rows<D, 4>(qrow + h * D, D, qd, p.q_norm_w, p.eps, lane, c, s);
            }
            for (; h < p.Hq; ++h) {
                __nv_bfloat16* qd[1] = {qrow + h * D};
                rope_rows<D, 1>(qrow + h * D, D, qd, p.q_norm_w, p.eps, lane, c, s);
            }
        }
        if (phys < 0 || phys >= p.num_pages) {
            if (lane == 0) report(p.status, PA_ERR_BAD_PAGE);
            continue;
        }
        // K heads (rotated) and V heads (copied), four at a time
        for (int g0 = 0; g0 < p.Hkv; g0 += 4) {
            const int nh = min(4, p.Hkv - g0);
            __nv_bfloat16* kd[4];
            float v1[4][PPL], v2[4][PPL];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int g = g0 + (h < nh ? h : 0);
                kd[h] = p.k_pool + (((size_t)phys * p.Hkv + g) * p.page_size + slot) * D;
                if (h < nh) PairIO<D>::load(p.v_new + ((size_t)t * p.Hkv + g) * D, lane, v1[h], v2[h]);
            }
            const __nv_bfloat16* ks = p.k_new + ((size_t)t * p.Hkv + g0) * D;
            if (nh == 4) {
                rope_rows<D, 4>(ks, D, kd, p.k_norm_w, p.eps, lane, c, s);
            } else {
                for (int h = 0; h < nh; ++h) rope_rows<D, 1>(ks + h * D, D, kd + h, p.k_norm_w, p.eps, lane, c, s);
            }
#pragma unroll
            for (int h = 0; h < 4; ++h)
                if (h < nh) PairIO<D>::store(kd[h] - p.k_pool + p.v_pool, lane, v1[h], v2[h]);  // exact copy
        }
    }
}

// One warp per new token; lane l quantises elements [l * D/32, (l+1) * D/32) of every head row.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) kv_write_fp8_kernel(
    uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, const float* __restrict__ k_scale, const float* __restrict__ v_scale,
    const int32_t* __restrict__ cu_new, const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
    int num_pages, int max_pages, int batch, int total_new, int page_size, int num_kv_heads, int32_t* status) {
    constexpr int EPL = D / 32;  // elements per lane (2 or 4)
    pdl_launch_dependents();  // the next kernel (e.g. the decode) may start; it waits for our writes
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * kWarps;
    for (int t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < total_new; t += nwarps) {
        const int b = find_seq(cu_new, batch, t);
        if (b < 0 || b >= batch) {
            if (lane == 0) report(status, PA_ERR_BAD_LEN);
            continue;
        }
        const int n_b = __ldg(cu_new + b + 1) - __ldg(cu_new + b);
        const int i = t - __ldg(cu_new + b);
        const int pos = __ldg(seq_lens + b) - n_b + i;
        if (n_b <= 0 || i >= n_b || pos < 0 || pos >= max_pages * page_size) {
            if (lane == 0) report(status, PA_ERR_BAD_LEN);
            continue;
        }
        const int phys = __ldg(block_table + (size_t)b * max_pages + pos / page_size);
        if (phys < 0 || phys >= num_pages) {
            if (lane == 0) report(status, PA_ERR_BAD_PAGE);
            continue;
        }
        const int slot = pos % page_size;
        for (int g = 0; g < num_kv_heads; ++g) {
            const float ks = __ldg(k_scale + g), vs = __ldg(v_scale + g);
            const size_t src = ((size_t)t * num_kv_heads + g) * D + lane * EPL;
            const size_t blk = (size_t)phys * num_kv_heads + g;
            float kx[EPL], vx[EPL];
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
                const __nv_bfloat162 kk = *reinterpret_cast<const __nv_bfloat162*>(k_new + src + e);
                const __nv_bfloat162 vv = *reinterpret_cast<const __nv_bfloat162*>(v_new + src + e);
                kx[e] = __low2float(kk) / ks;
                kx[e + 1] = __high2float(kk) / ks;
                vx[e] = __low2float(vv) / vs;
                vx[e + 1] = __high2float(vv) / vs;
            }
            uint32_t kcodes = 0;
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
                const uint32_t kc = __nv_cvt_float2_to_fp8x2(make_float2(kx[e], kx[e + 1]), __NV_SATFINITE, __NV_E4M3);
                const uint32_t vc = __nv_cvt_float2_to_fp8x2(make_float2(vx[e], vx[e + 1]), __NV_SATFINITE, __NV_E4M3);
                kcodes |= (kc & 0xFFFFu) << (8 * e);
                // V is transposed: element d of the row goes to row d of the page block, column slot
                uint8_t* vcol = v_pool + (blk * D + lane * EPL + e) * page_size + slot;
                vcol[0] = (uint8_t)(vc & 0xFF);
                vcol[page_size] = (uint8_t)((vc >> 8) & 0xFF);
            }
            uint8_t* krow = k_pool + (blk * page_size + slot) * D + lane * EPL;
            if constexpr (EPL == 4)
                *reinterpret_cast<uint32_t*>(krow) = kcodes;
            else
                *reinterpret_cast<uint16_t*>(krow) = (uint16_t)kcodes;
        }
    }
}

}  // namespace kvw
}  // namespace pa

extern "C" int kv_write_paged(void* k_pool, void* v_pool, int num_pages, const void* k_new, const void* v_new,
                              const int32_t* cu_seqlens_new, const int32_t* seq_lens, const int32_t* block_table,
                              int max_pages_per_seq, int batch, int total_new, int page_size, int num_kv_heads,
                              int head_dim, int32_t* status, void* stream) {
    using namespace pa;
    NvtxRange nvtx_("kv_write_paged");
    if (batch < 0 || total_new < 0) return PA_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_SHAPE;
    if (page_size < 16 || page_size > 256 || page_size % 16 != 0) return PA_ERR_SHAPE;
    if (num_kv_heads < 1) return PA_ERR_SHAPE;
    if (batch == 0 || total_new == 0) return PA_OK;
    if (!k_pool || !v_pool || !k_new || !v_new || !cu_seqlens_new || !seq_lens || !block_table) return PA_ERR_NULL;
    if (num_pages < 1 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_SHAPE;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != PA_OK) return rc;
    const int blocks_needed = (total_new + 2 * kvw::kWarps - 1) / (2 * kvw::kWarps);  // two rows per warp
    const int grid = blocks_needed < dev.sm_count * 16 ? blocks_needed : dev.sm_count * 16;
    log_config("kv writeback: head_dim %d, two new rows per warp at a time, grid %d CTAs x %d warps", head_dim, grid,
               kvw::kWarps);
    kvw::kv_write_kernel<<<grid, kvw::kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<__nv_bfloat16*>(k_pool), static_cast<__nv_bfloat16*>(v_pool),
        static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), cu_seqlens_new, seq_lens,
        block_table, num_pages, max_pages_per_seq, batch, total_new, page_size, num_kv_heads, head_dim, status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" int kv_write_paged_rope(void* k_pool, void* v_pool, int num_pages, const void* k_new, const void* v_new,
                                   void* q, int num_q_heads, const int32_t* cu_seqlens_new, const int32_t* seq_lens,
                                   const int32_t* block_table, int max_pages_per_seq, int batch, int total_new,
                                   int page_size, int num_kv_heads, int head_dim, float rope_base,
                                   const void* q_norm_weight, const void* k_norm_weight, float norm_eps,
                                   int32_t* status, void* stream) {
    using namespace pa;
    NvtxRange nvtx_("kv_write_paged_rope");
    if (batch < 0 || total_new < 0) return PA_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_SHAPE;
    if (page_size < 16 || page_size > 256 || page_size % 16 != 0) return PA_ERR_SHAPE;
    if (num_kv_heads < 1) return PA_ERR_SHAPE;
    if (q != nullptr && (num_q_heads < num_kv_heads || num_q_heads % num_kv_heads != 0)) return PA_ERR_SHAPE;
    if (!(rope_base > 1.f) || rope_base == INFINITY) return PA_ERR_SHAPE;  // also rejects NaN
    if (!(norm_eps >= 0.f) || norm_eps == INFINITY) return PA_ERR_SHAPE;
    if (batch == 0 || total_new == 0) return PA_OK;
    if (!k_pool || !v_pool || !k_new || !v_new || !cu_seqlens_new || !seq_lens || !block_table) return PA_ERR_NULL;
    if (num_pages < 1 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_SHAPE;
    if ((q && !aligned16(q)) || (q_norm_weight && !aligned16(q_norm_weight)) ||
        (k_norm_weight && !aligned16(k_norm_weight)))
        return PA_ERR_SHAPE;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != PA_OK) return rc;

    kvw::RopeParams prm;
    prm.k_pool = static_cast<__nv_bfloat16*>(k_pool);
    prm.v_pool = static_cast<__nv_bfloat16*>(v_pool);
    prm.k_new = static_cast<const __nv_bfloat16*>(k_new);
    prm.v_new = static_cast<const __nv_bfloat16*>(v_new);
    prm.q = static_cast<__nv_bfloat16*>(q);
    prm.q_norm_w = static_cast<const __nv_bfloat16*>(q_norm_weight);
    prm.k_norm_w = static_cast<const __nv_bfloat16*>(k_norm_weight);
    prm.cu_new = cu_seqlens_new;
    prm.seq_lens = seq_lens;
    prm.block_table = block_table;
    prm.status = status;
    prm.num_pages = num_pages;
    prm.max_pages = max_pages_per_seq;
    prm.batch = batch;
    prm.total_new = total_new;
    prm.page_size = page_size;
    prm.Hkv = num_kv_heads;
    prm.Hq = q != nullptr ? num_q_heads : 0;
    prm.eps = norm_eps;
    // frequencies as 64-bit fractions of a turn: theta_i = base^(-2i/D) <= 1 rad < 1 turn
    for (int i = 0; i < 64; ++i) {
        if (i < head_dim / 2) {
            const double theta = std::pow((double)rope_base, -2.0 * i / head_dim);
            const double turns = theta / (2.0 * M_PI);  // in (0, 0.16]
            prm.turns[i] = (unsigned long long)(turns * 18446744073709551616.0);
        } else {
            prm.turns[i] = 0;
        }
    }
    const int blocks_needed = (total_new + kvw::kWarps - 1) / kvw::kWarps;
    const int grid = blocks_needed < dev.sm_count * 16 ? blocks_needed : dev.sm_count * 16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    log_config("kv writeback with RoPE%s%s: head_dim %d, grid %d CTAs x %d warps", k_norm_weight ? " + K norm" : "",
               q ? " (+ queries in place)" : "", head_dim, grid, kvw::kWarps);
    if (head_dim == 128)
        kvw::kv_write_rope_kernel<128><<<grid, kvw::kWarps * 32, 0, st>>>(prm);
    else
        kvw::kv_write_rope_kernel<64><<<grid, kvw::kWarps * 32, 0, st>>>(prm);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" int kv_write_paged_fp8(void* k_pool, void* v_pool, int num_pages, const void* k_new, const void* v_new,
                                  const float* k_scale, const float* v_scale, const int32_t* cu_seqlens_new,
                                  const int32_t* seq_lens, const int32_t* block_table, int max_pages_per_seq,
                                  int batch, int total_new, int page_size, int num_kv_heads, int head_dim,
                                  int32_t* status, void* stream) {
    using namespace pa;
    NvtxRange nvtx_("kv_write_paged_fp8");
    if (batch < 0 || total_new < 0) return PA_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_SHAPE;
    if (page_size < 16 || page_size > 256 || (page_size & (page_size - 1)) != 0) return PA_ERR_SHAPE;
    if (num_kv_heads < 1) return PA_ERR_SHAPE;
    if (batch == 0 || total_new == 0) return PA_OK;
    if (!k_pool || !v_pool || !k_new || !v_new || !k_scale || !v_scale || !cu_seqlens_new || !seq_lens ||
        !block_table)
        return PA_ERR_NULL;
    if (num_pages < 1 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_SHAPE;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != PA_OK) return rc;
    const int blocks_needed = (total_new + kvw::kWarps - 1) / kvw::kWarps;
    const int grid = blocks_needed < dev.sm_count * 16 ? blocks_needed : dev.sm_count * 16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto* kp = static_cast<uint8_t*>(k_pool);
    auto* vp = static_cast<uint8_t*>(v_pool);
    auto* kn = static_cast<const __nv_bfloat16*>(k_new);
    auto* vn = static_cast<const __nv_bfloat16*>(v_new);
    log_config("kv writeback to fp8 e4m3: head_dim %d, grid %d CTAs x %d warps", head_dim, grid, kvw::kWarps);
    if (head_dim == 128)
        kvw::kv_write_fp8_kernel<128><<<grid, kvw::kWarps * 32, 0, st>>>(
            kp, vp, kn, vn, k_scale, v_scale, cu_seqlens_new, seq_lens, block_table, num_pages, max_pages_per_seq,
            batch, total_new, page_size, num_kv_heads, status);
    else
        kvw::kv_write_fp8_kernel<64><<<grid, kvw::kWarps * 32, 0, st>>>(
            kp, vp, kn, vn, k_scale, v_scale, cu_seqlens_new, seq_lens, block_table, num_pages, max_pages_per_seq,
            batch, total_new, page_size, num_kv_heads, status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
