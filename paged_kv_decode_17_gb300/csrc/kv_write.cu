// Eager K/V writeback into pages ("Inside Ion", section "IonAttention in One
// Paragraph": KV pages are written back eagerly as they are produced).
//
// One warp per new token: it finds the token's sequence by binary search
// over cu_seqlens_new, resolves (page, slot) through the block table, and
// copies the token's [Hkv][D] K and V rows with 16-byte vector loads and
// stores.  A bit-exact copy; nothing else in the pools is written.
#include "pa_common.cuh"
#include "pa_host.h"

namespace pa {
namespace kvw {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) kv_write_kernel(
    __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ v_pool, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, const int32_t* __restrict__ cu_new, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, int num_pages, int max_pages, int batch, int total_new, int page_size,
    int num_kv_heads, int head_dim, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int vec_per_head = head_dim / 8;  // 16-byte vectors per row
    const int vec_per_tok = num_kv_heads * vec_per_head;
    const int nwarps = gridDim.x * kWarps;
    for (int t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < total_new; t += nwarps) {
        // sequence of token t: largest b with cu_new[b] <= t (skipping empty ones)
        int lo = 0, hi = batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(cu_new + mid) <= t) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int n_b = __ldg(cu_new + b + 1) - __ldg(cu_new + b);
        const int i = t - __ldg(cu_new + b);
        const int L = __ldg(seq_lens + b);
        const int pos = L - n_b + i;
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
        const uint4* ks = reinterpret_cast<const uint4*>(k_new + (size_t)t * num_kv_heads * head_dim);
        const uint4* vs = reinterpret_cast<const uint4*>(v_new + (size_t)t * num_kv_heads * head_dim);
        for (int v = lane; v < vec_per_tok; v += 32) {
            const int g = v / vec_per_head;
            const int c = v - g * vec_per_head;
            const size_t dst = (((size_t)phys * num_kv_heads + g) * page_size + slot) * head_dim / 8 + c;
            const uint4 kv = __ldg(ks + v);
            const uint4 vv = __ldg(vs + v);
            reinterpret_cast<uint4*>(k_pool)[dst] = kv;
            reinterpret_cast<uint4*>(v_pool)[dst] = vv;
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
    const int blocks_needed = (total_new + kvw::kWarps - 1) / kvw::kWarps;
    const int grid = blocks_needed < dev.sm_count * 16 ? blocks_needed : dev.sm_count * 16;
    kvw::kv_write_kernel<<<grid, kvw::kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<__nv_bfloat16*>(k_pool), static_cast<__nv_bfloat16*>(v_pool),
        static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), cu_seqlens_new, seq_lens,
        block_table, num_pages, max_pages_per_seq, batch, total_new, page_size, num_kv_heads, head_dim, status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
