// Varlen causal prefill: plan kernel, host launcher and C-ABI entry point.  The
// main kernel and its design are in prefill_dev.cuh.
#include "prefill_dev.cuh"
#include "pa_trace.h"

#include <algorithm>
#include <mutex>

namespace pa {
namespace pf {

// ---------------------------------------------------------------------------------- plan
// List every (sequence, query tile) of entries with q_len > kDecodeMaxQ, sorted by the number
// of 128-key tiles the tile attends (counting sort, heaviest first).  One CTA.
__global__ void __launch_bounds__(PLAN_THREADS) prefill_plan_kernel(const int32_t* __restrict__ cu_q,
                                                                     const int32_t* __restrict__ seq_lens,
                                                                     int batch, int cap, int max_cost, int2* tiles,
                                                                     int32_t* n_tiles, int32_t* status) {
    extern __shared__ int hist[];  // [max_cost + 1] counts, then running offsets
    __shared__ int s_total;
    for (int c = threadIdx.x; c <= max_cost; c += blockDim.x) hist[c] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        int ql, sl;
        const int nt = seq_tiles(cu_q, seq_lens, b, cap, status, ql, sl);
        for (int t = 0; t < nt; ++t) {
            const int rows = min(BM, ql - t * BM);
            const int cost = min(max_cost, (sl - ql + t * BM + rows - 1) / BN + 1);
            atomicAdd(&hist[cost], 1);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // exclusive offsets, heaviest cost first
        int run = 0;
        for (int c = max_cost; c >= 0; --c) {
            const int n = hist[c];
            hist[c] = run;
            run += n;
        }
        s_total = run;
    }
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        int ql, sl;
        const int nt = seq_tiles(cu_q, seq_lens, b, cap, nullptr, ql, sl);
        for (int t = 0; t < nt; ++t) {
            const int rows = min(BM, ql - t * BM);
            const int cost = min(max_cost, (sl - ql + t * BM + rows - 1) / BN + 1);
            tiles[atomicAdd(&hist[cost], 1)] = make_int2(b, t);
        }
    }
    if (threadIdx.x == 0) *n_tiles = s_total;
}

}  // namespace pf
}  // namespace pa

using namespace pa;

extern "C" size_t pa_prefill_workspace_bytes(int batch, int total_q, int num_q_heads, int num_kv_heads,
                                             int head_dim) {
    const size_t dec = pa_decode_multiquery_workspace_bytes(batch, kDecodeMaxQ, num_q_heads, num_kv_heads, head_dim);
    if (dec == 0 || total_q < 0) return 0;
    return align_up(dec, 256) + pf::plan_bytes(batch, total_q);
}

namespace {
// CTAs of the prefill kernel that can be resident at once (queried once per device / variant).
std::mutex g_occ_mu;
int g_occ[64][3] = {};

template <int D, bool PAIR>
int max_ctas(int device, cudaLaunchConfig_t cfg) {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (device < 0 || device >= 64) return 0;
    int& v = g_occ[device][PAIR ? 2 : (D == 128 ? 1 : 0)];
    if (v == 0) {
        if (PAIR) {
            int n = 0;
            cfg.gridDim = dim3(2, 1, 1);
            if (cudaOccupancyMaxActiveClusters(&n, pf::prefill_kernel<D, PAIR>, &cfg) != cudaSuccess || n <= 0)
                return 0;
            v = 2 * n;
        } else {
            int per_sm = 0, sms = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pf::prefill_kernel<D, PAIR>, pf::NTHREADS,
                                                              pf::Cfg<D, PAIR>::SMEM_BYTES) != cudaSuccess ||
                per_sm <= 0)
                return 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
                return 0;
            v = per_sm * sms;
        }
    }
    return v;
}

template <int D, bool PAIR>
int launch_persistent(cudaStream_t st, int device, long long items_upper, const CUtensorMap& qmap,
                      const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& omap,
                      const pf::Params& prm) {
    using C = pf::Cfg<D, PAIR>;
    if (set_smem_limit_once((const void*)pf::prefill_kernel<D, PAIR>, C::SMEM_BYTES, device,
                            PAIR ? 19 : (D == 128 ? 2 : 3)) != PA_OK)
        return PA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(pf::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PAIR ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 1 : 0;
    long long n = max_ctas<D, PAIR>(device, cfg);
    if (n <= 0) return PA_ERR_CUDA;
    const long long units = PAIR ? 2 * items_upper : items_upper;  // a pair works on one item at a time
    if (n > units) n = units;
    if (PAIR) n &= ~1ll;
    cfg.gridDim = dim3((unsigned)n, 1, 1);
    log_config("varlen causal prefill: head_dim %d, persistent grid %lld CTAs x %d threads (1 per SM)%s, "
               "query tile %d rows x key tile %d, %s, K ring %d / V ring %d stages, %d B smem",
               D, n, pf::NTHREADS, PAIR ? " in CTA pairs (one M = 256 MMA per tile, cta_group::2)" : "",
               pf::BM, pf::BN, PAIR ? "4 heads per pair" : "2 heads per CTA", C::NKr, C::NVr, C::SMEM_BYTES);
    return cudaLaunchKernelEx(&cfg, pf::prefill_kernel<D, PAIR>, qmap, kmap, vmap, omap, prm) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}
}  // namespace

extern "C" int attn_prefill_varlen_causal(void* out, float* lse, const void* q, const void* k_pool,
                                          const void* v_pool, int num_pages, const int32_t* block_table,
                                          int max_pages_per_seq, const int32_t* cu_seqlens_q,
                                          const int32_t* seq_lens, int batch, int total_q, int max_q_len,
                                          int max_seq_len, int page_size, int num_q_heads, int num_kv_heads,
                                          int head_dim, float softmax_scale, void* workspace,
                                          size_t workspace_bytes, int32_t* status, void* stream) {
    NvtxRange nvtx_("attn_prefill_varlen_causal");
    if (batch < 0 || total_q < 0 || max_q_len < 0 || max_seq_len < 0) return PA_ERR_SHAPE;
    int rc = check_common_shapes(page_size, num_q_heads, num_kv_heads, head_dim);
    if (rc != PA_OK) return rc;
    if (!(softmax_scale > 0.f) || softmax_scale == INFINITY) return PA_ERR_SHAPE;  // also rejects NaN
    if (batch == 0 || total_q == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_table || !cu_seqlens_q || !seq_lens) return PA_ERR_NULL;
    if (num_pages < 1 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
    if ((long long)max_seq_len > (long long)max_pages_per_seq * page_size) return PA_ERR_SHAPE;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(q) || !aligned16(out)) return PA_ERR_SHAPE;
    const long long pool_rows = (long long)num_pages * num_kv_heads * page_size;
    if (pool_rows >= (1ll << 31)) return PA_ERR_SHAPE;

    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc != PA_OK) return rc;

    const size_t need = pa_prefill_workspace_bytes(batch, total_q, num_q_heads, num_kv_heads, head_dim);
    if (workspace == nullptr || need == 0) return PA_ERR_WORKSPACE;
    if (workspace_bytes < need) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_WORKSPACE;
    const size_t dec_bytes =
        pa_decode_multiquery_workspace_bytes(batch, kDecodeMaxQ, num_q_heads, num_kv_heads, head_dim);

    // entries with q_len <= kDecodeMaxQ: split-K decode over their KV
    const int dec_qmax = max_q_len < 1 ? 1 : (max_q_len < kDecodeMaxQ ? max_q_len : kDecodeMaxQ);
    if (max_q_len <= kDecodeMaxQ)  // no entry needs the prefill kernel
        return dec::launch_decode(out, lse, q, k_pool, v_pool, num_pages, block_table, max_pages_per_seq, seq_lens,
                                  cu_seqlens_q, total_q, dec_qmax, kDecodeMaxQ, batch, max_seq_len, page_size,
                                  num_q_heads, num_kv_heads, head_dim, softmax_scale, workspace, dec_bytes, status,
                                  stream, /*per_segment=*/true);

    const int group = num_q_heads / num_kv_heads;
    // CTA pairs (one M = 256 MMA per tile over two SMs) only when asked for: measured on the
    // 16 x 512..4096-token prefill (Hq 28, Hkv 4) they took 1.11 ms against 0.74 ms for single
    // CTAs -- every tile's softmax / MMA hand-over (scores freed, P ready, MMA done) then
    // crosses SMs, and with one S and one P buffer per head that latency is on the critical path
    const bool pair = head_dim == 128 && prefill_pair_override() == 1;
    const int NPC = (group + 1) / 2;  // head pairs per KV head (single CTAs; the fused kernel)
    const int NPC_PAIR = (group + 3) / 4;  // blocks of 4 heads per KV head (CTA pairs)
    const long long tiles_upper = (long long)(total_q + pf::BM - 1) / pf::BM + batch;
    const long long items_upper = tiles_upper * num_kv_heads * NPC;
    const long long items_upper_pair = tiles_upper * num_kv_heads * NPC_PAIR;

    // plan: query tiles sorted by cost
    const pf::PlanArea plan = pf::plan_area(static_cast<uint8_t*>(workspace) + align_up(dec_bytes, 256));
    const int max_cost = (int)std::min<long long>((long long)max_seq_len / pf::BN + 1, pf::PLAN_MAX_COST);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    CUtensorMap qmap, kmap, vmap, omap;
    if (encode_q_map(&qmap, q, total_q, num_q_heads, head_dim) != PA_OK) return PA_ERR_CUDA;
    if (encode_q_map(&omap, out, total_q, num_q_heads, head_dim) != PA_OK) return PA_ERR_CUDA;
    if (head_dim == 128 && !pair) {  // one TMA box per 16-key page block (pf::Cfg::BLK4)
        if (encode_blocks_map(&kmap, k_pool, (uint64_t)pool_rows / 16) != PA_OK) return PA_ERR_CUDA;
        if (encode_blocks_map(&vmap, v_pool, (uint64_t)pool_rows / 16) != PA_OK) return PA_ERR_CUDA;
    } else {
        if (encode_rows_map(&kmap, k_pool, (uint64_t)pool_rows, head_dim, 64, 16) != PA_OK) return PA_ERR_CUDA;
        if (encode_rows_map(&vmap, v_pool, (uint64_t)pool_rows, head_dim, 64, 16) != PA_OK) return PA_ERR_CUDA;
    }

    pf::Params prm;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.block_table = block_table;
    prm.seq_lens = seq_lens;
    prm.cu_q = cu_seqlens_q;
    prm.tiles = plan.tiles;
    prm.n_tiles = plan.n_tiles;
    prm.status = status;
    prm.num_pages = num_pages;
    prm.max_pages = max_pages_per_seq;
    prm.batch = batch;
    prm.page_size = page_size;
    prm.Hq = num_q_heads;
    prm.Hkv = num_kv_heads;
    prm.group = group;
    prm.NPC = NPC;
    prm.scale_log2 = softmax_scale * kLog2e;
    prm.wait_ns = prefill_wait_ns(kWaitTimeoutNs);

    // one persistent launch for the decode rows and the prefill tiles (+ the merge of split decode rows)
    if (prefill_path_override() != 2)
        return pf::launch_fused(head_dim, st, out, lse, q, k_pool, v_pool, num_pages, block_table, max_pages_per_seq,
                                cu_seqlens_q, seq_lens, batch, total_q, max_seq_len, page_size, num_q_heads,
                                num_kv_heads, softmax_scale, workspace, dec_bytes, status, qmap, kmap, vmap, omap, prm,
                                plan, max_cost);

    // separate kernels: split-K decode (+ merge), plan, prefill
    rc = dec::launch_decode(out, lse, q, k_pool, v_pool, num_pages, block_table, max_pages_per_seq, seq_lens,
                            cu_seqlens_q, total_q, dec_qmax, kDecodeMaxQ, batch, max_seq_len, page_size,
                            num_q_heads, num_kv_heads, head_dim, softmax_scale, workspace, dec_bytes, status,
                            stream, /*per_segment=*/true);
    if (rc != PA_OK) return rc;
    const int plan_smem = (max_cost + 1) * (int)sizeof(int);
    if (set_smem_limit_once((const void*)pf::prefill_plan_kernel, 48 * 1024, dev.device, 4) != PA_OK)
        return PA_ERR_CUDA;
    pf::prefill_plan_kernel<<<1, pf::PLAN_THREADS, plan_smem, st>>>(
        cu_seqlens_q, seq_lens, batch, max_pages_per_seq * page_size, max_cost, plan.tiles, plan.n_tiles, status);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (pair) {
        prm.NPC = NPC_PAIR;
        return launch_persistent<128, true>(st, dev.device, items_upper_pair, qmap, kmap, vmap, omap, prm);
    }
    if (head_dim == 128)
        return launch_persistent<128, false>(st, dev.device, items_upper, qmap, kmap, vmap, omap, prm);
    return launch_persistent<64, false>(st, dev.device, items_upper, qmap, kmap, vmap, omap, prm);
}
