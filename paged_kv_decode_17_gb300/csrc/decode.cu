// Split-K paged decode: host launchers and C-ABI entry points.  The kernels
// and their design are in decode_dev.cuh.
#include "decode_dev.cuh"
#include "pa_trace.h"

#include <climits>
#include <mutex>

using namespace pa;

extern "C" size_t pa_decode_multiquery_workspace_bytes(int batch, int max_q_len, int num_q_heads, int num_kv_heads,
                                                       int head_dim) {
    if (batch <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads) return 0;
    if (max_q_len < 1 || max_q_len > kDecodeMaxQ || num_q_heads / num_kv_heads > 128) return 0;
    DeviceInfo dev;
    if (current_device(&dev) != PA_OK) return 0;
    return dec::ws_bytes(dev.sm_count, batch, num_q_heads, num_kv_heads, head_dim, max_q_len);
}

extern "C" size_t pa_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim) {
    return pa_decode_multiquery_workspace_bytes(batch, 1, num_q_heads, num_kv_heads, head_dim);
}

namespace pa {
namespace dec {

// Check the arguments of a split-K decode and fill in its launch: parameters, grid,
// variant.  cu_q == nullptr: one query row per sequence
// (row b).  Otherwise entries with 1 <= q_len <= qmax are served (rows
// cu_q[b] ..), q_len in (qmax, qcap] is reported as PA_ERR_BAD_LEN and
// longer entries are left to the prefill kernel.
// k_scale / v_scale non-null: the pools hold e4m3 codes (V transposed per page block).
// per_segment: when not every segment fits the swapped-operand variant, choose the
// operand order per segment (bf16, no append) instead of the plain order everywhere.
// grid_override > 0: the number of (virtual) CTAs that will run the decode body.
// L->grid == 0 on return: nothing to launch.
int prepare_decode(DecodeLaunch* L, void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                            const float* k_scale, const float* v_scale, const void* k_new, const void* v_new,
                            int num_pages, const int32_t* block_table,
                            int max_pages_per_seq, const int32_t* seq_lens, const int32_t* cu_q, int total_q,
                            int qmax, int qcap, int batch, int max_seq_len, int page_size, int num_q_heads,
                            int num_kv_heads, int head_dim, float softmax_scale, void* workspace,
                            size_t workspace_bytes, int32_t* status, bool per_segment, int grid_override) {
    const bool fp8 = k_scale != nullptr;
    if (batch < 0 || max_seq_len < 0 || total_q < 0) return PA_ERR_SHAPE;
    if (qmax < 1 || qmax > kDecodeMaxQ || (cu_q == nullptr && qmax != 1)) return PA_ERR_SHAPE;
    int rc = check_common_shapes(page_size, num_q_heads, num_kv_heads, head_dim);
    if (rc != PA_OK) return rc;
    L->grid = 0;
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_table || !seq_lens) return PA_ERR_NULL;
    if (num_pages < 1 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
    if ((long long)max_seq_len > (long long)max_pages_per_seq * page_size) return PA_ERR_SHAPE;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(q) || !aligned16(out)) return PA_ERR_SHAPE;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_NULL;
    if (k_new != nullptr && (fp8 || !aligned16(k_new) || !aligned16(v_new))) return PA_ERR_SHAPE;
    const long long pool_rows = (long long)num_pages * num_kv_heads * page_size;
    if (pool_rows >= (1ll << 31)) return PA_ERR_SHAPE;

    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc != PA_OK) return rc;

    const int group = num_q_heads / num_kv_heads;
    const Bounds bd = bounds(group, qmax);
    const int nrb_max = bd.RS / RB;
    const long long segs = (long long)batch * num_kv_heads * bd.SBmax;
    const long long units_upper = segs * nrb_max * ((max_seq_len + UNIT - 1) / UNIT);
    const int min_chunk = decode_min_chunk(MIN_CHUNK);
    // every unit index and grid * chunk must fit in int32
    if (segs * nrb_max * ((max_pages_per_seq * (long long)page_size + UNIT - 1) / UNIT) +
            (long long)dev.sm_count * kMaxCtasPerSM * min_chunk >=
        (1ll << 31))
        return PA_ERR_SHAPE;
    const bool swap = group * qmax <= 8;  // at most 8 rows per segment: the swapped-operand variant
    // some segments (the one-row entries) may fit it
    const bool mixed_order = per_segment && !swap && group <= 8 && !fp8 && k_new == nullptr;
    const int gmax = dev.sm_count * ((fp8 && swap) ? ctas_per_sm<true, true>() : ctas_per_sm<false, false>());
    long long g = (units_upper + min_chunk - 1) / min_chunk;
    if (g < 1) g = 1;
    const int grid = grid_override > 0 ? grid_override : (int)(g < gmax ? g : gmax);
    if (grid > dev.sm_count * kMaxCtasPerSM) return PA_ERR_SHAPE;  // workspace slots are sized for that many

    const WsLayout wl = ws_layout(ws_slots(dev.sm_count, (int)segs), batch, bd.RS, head_dim);  // as *_workspace_bytes
    if (workspace == nullptr) return PA_ERR_WORKSPACE;
    if (workspace_bytes < wl.total) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_WORKSPACE;
    dec::Params prm;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
    prm.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
    prm.k_scale = k_scale;
    prm.v_scale = v_scale;
    prm.k_new = static_cast<const __nv_bfloat16*>(k_new);
    prm.v_new = static_cast<const __nv_bfloat16*>(v_new);
    prm.k_pool_w = k_new != nullptr ? static_cast<__nv_bfloat16*>(const_cast<void*>(k_pool)) : nullptr;
    prm.v_pool_w = k_new != nullptr ? static_cast<__nv_bfloat16*>(const_cast<void*>(v_pool)) : nullptr;
    prm.block_table = block_table;
    prm.seq_lens = seq_lens;
    prm.cu_q = cu_q;
    prm.total_q = cu_q == nullptr ? batch : total_q;
    prm.qmax = qmax;
    prm.qcap = qcap;
    prm.SBmax = bd.SBmax;
    prm.RS = bd.RS;
    prm.min_chunk = min_chunk;
    prm.reset_words = nullptr;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    prm.seg_base = reinterpret_cast<int32_t*>(ws + wl.hdr);
    prm.G = grid;
    prm.ws_lse = reinterpret_cast<float*>(ws + wl.lse);
    prm.ws_o = reinterpret_cast<float*>(ws + wl.o);
    prm.status = status;
    prm.num_pages = num_pages;
    prm.max_pages = max_pages_per_seq;
    prm.batch = batch;
    prm.page_size = page_size;
    prm.ps_shift = __builtin_ctz((unsigned)page_size);
    prm.Hq = num_q_heads;
    prm.Hkv = num_kv_heads;
    prm.group = group;
    prm.scale_log2 = softmax_scale * kLog2e;

    L->prm = prm;
    L->grid = grid;
    L->segs = segs;
    L->nrb_max = nrb_max;
    L->head_dim = head_dim;
    L->device = dev.device;
    L->fp8 = fp8;
    L->swap = swap;
    L->mixed_order = mixed_order;
    L->app = k_new != nullptr;
    L->min_chunk = min_chunk;
    L->qmax = qmax;
    return PA_OK;
}

int launch_merge(const DecodeLaunch& L, cudaStream_t st) {
    // the merge of split segments, a programmatic dependent of the decode grid
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)L.segs, (unsigned)L.nrb_max, 1);
    cfg.blockDim = dim3(RB * L.head_dim / 4, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = L.head_dim == 128 ? cudaLaunchKernelEx(&cfg, merge_kernel<128>, L.prm)
                                            : cudaLaunchKernelEx(&cfg, merge_kernel<64>, L.prm);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

static int launch_decode_kv(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                            const float* k_scale, const float* v_scale, const void* k_new, const void* v_new,
                            int num_pages, const int32_t* block_table,
                            int max_pages_per_seq, const int32_t* seq_lens, const int32_t* cu_q, int total_q,
                            int qmax, int qcap, int batch, int max_seq_len, int page_size, int num_q_heads,
                            int num_kv_heads, int head_dim, float softmax_scale, void* workspace,
                            size_t workspace_bytes, int32_t* status, void* stream, bool per_segment = false) {
    DecodeLaunch L;
    int rc = prepare_decode(&L, out, lse, q, k_pool, v_pool, k_scale, v_scale, k_new, v_new, num_pages, block_table,
                            max_pages_per_seq, seq_lens, cu_q, total_q, qmax, qcap, batch, max_seq_len, page_size,
                            num_q_heads, num_kv_heads, head_dim, softmax_scale, workspace, workspace_bytes, status,
                            per_segment, 0);
    if (rc != PA_OK || L.grid == 0) return rc;
    const Params& prm = L.prm;
    const int grid = L.grid;
    const bool fp8 = L.fp8, swap = L.swap, mixed_order = L.mixed_order, app = L.app;
    const int min_chunk = L.min_chunk;
    const long long segs = L.segs;
    const int nrb_max = L.nrb_max;
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc != PA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto go = [&](auto kernel, int smem, int slot) {
        if (set_smem_limit_once((const void*)kernel, smem, dev.device, slot) != PA_OK) return PA_ERR_CUDA;
        // programmatic dependent launch: the CTAs may start (and set up) while the previous
        // kernel finishes; they wait for it in the kernel before touching any input
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(W * 32, 1, 1);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, prm) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    };
    log_config("split-K decode: head_dim %d, %s, operand order %s, %s, q_len <= %d, grid %d CTAs x %d warps "
               "(%d per SM), min chunk %d units of %d keys, merge grid %lld x %d",
               head_dim, fp8 ? "fp8 e4m3 pools" : "bf16 pools",
               swap ? "swapped (keys as M)" : (mixed_order ? "per segment" : "plain (query rows as M)"),
               app ? "newest rows appended in-kernel" : "no append", qmax, grid, W,
               (fp8 && swap) ? ctas_per_sm<true, true>() : ctas_per_sm<false, false>(), min_chunk, UNIT, segs,
               nrb_max);
    if (head_dim == 128) {
        if (fp8)
            rc = swap ? go(decode_kernel<128, true, true, false>, Cfg<128, true, true>::SMEM_BYTES, 7)
                      : go(decode_kernel<128, true, false, false>, Cfg<128, true, false>::SMEM_BYTES, 5);
        else if (app)
            rc = swap ? go(decode_kernel<128, false, true, true>, Cfg<128, false, true>::SMEM_BYTES, 11)
                      : go(decode_kernel<128, false, false, true>, Cfg<128, false, false>::SMEM_BYTES, 12);
        else if (mixed_order)
            rc = go(decode_kernel<128, false, 2, false>, Cfg<128, false, false>::SMEM_BYTES, 15);
        else
            rc = swap ? go(decode_kernel<128, false, true, false>, Cfg<128, false, true>::SMEM_BYTES, 8)
                      : go(decode_kernel<128, false, false, false>, Cfg<128, false, false>::SMEM_BYTES, 0);
    } else {
        if (fp8)
            rc = swap ? go(decode_kernel<64, true, true, false>, Cfg<64, true, true>::SMEM_BYTES, 9)
                      : go(decode_kernel<64, true, false, false>, Cfg<64, true, false>::SMEM_BYTES, 6);
        else if (app)
            rc = swap ? go(decode_kernel<64, false, true, true>, Cfg<64, false, true>::SMEM_BYTES, 13)
                      : go(decode_kernel<64, false, false, true>, Cfg<64, false, false>::SMEM_BYTES, 14);
        else if (mixed_order)
            rc = go(decode_kernel<64, false, 2, false>, Cfg<64, false, false>::SMEM_BYTES, 16);
        else
            rc = swap ? go(decode_kernel<64, false, true, false>, Cfg<64, false, true>::SMEM_BYTES, 10)
                      : go(decode_kernel<64, false, false, false>, Cfg<64, false, false>::SMEM_BYTES, 1);
    }
    if (rc != PA_OK) return rc;
    rc = launch_merge(L, st);
    if (rc != PA_OK) return rc;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_decode(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool, int num_pages,
                  const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                  const int32_t* cu_q, int total_q, int qmax, int qcap, int batch, int max_seq_len, int page_size,
                  int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale, void* workspace,
                  size_t workspace_bytes, int32_t* status, void* stream, bool per_segment) {
    return launch_decode_kv(out, lse, q, k_pool, v_pool, nullptr, nullptr, nullptr, nullptr, num_pages, block_table,
                            max_pages_per_seq, seq_lens, cu_q, total_q, qmax, qcap, batch, max_seq_len, page_size,
                            num_q_heads, num_kv_heads, head_dim, softmax_scale, workspace, workspace_bytes, status,
                            stream, per_segment);
}

}  // namespace dec
}  // namespace pa

extern "C" int attn_decode_paged_fp8(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                                     const float* k_scale, const float* v_scale, int num_pages,
                                     const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                                     int batch, int max_seq_len, int page_size, int num_q_heads, int num_kv_heads,
                                     int head_dim, float softmax_scale, void* workspace, size_t workspace_bytes,
                                     int32_t* status, void* stream) {
    NvtxRange nvtx_("attn_decode_paged_fp8");
    if (batch > 0 && (k_scale == nullptr || v_scale == nullptr)) return PA_ERR_NULL;
    return dec::launch_decode_kv(out, lse, q, k_pool, v_pool, k_scale, v_scale, nullptr, nullptr, num_pages,
                                 block_table, max_pages_per_seq, seq_lens, nullptr, batch, 1, 1, batch, max_seq_len,
                                 page_size, num_q_heads, num_kv_heads, head_dim, softmax_scale, workspace,
                                 workspace_bytes, status, stream);
}

extern "C" int attn_decode_paged(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                                 int num_pages, const int32_t* block_table, int max_pages_per_seq,
                                 const int32_t* seq_lens, int batch, int max_seq_len, int page_size, int num_q_heads,
                                 int num_kv_heads, int head_dim, float softmax_scale, void* workspace,
                                 size_t workspace_bytes, int32_t* status, void* stream) {
    NvtxRange nvtx_("attn_decode_paged");
    return dec::launch_decode(out, lse, q, k_pool, v_pool, num_pages, block_table, max_pages_per_seq, seq_lens,
                              nullptr, batch, 1, 1, batch, max_seq_len, page_size, num_q_heads, num_kv_heads,
                              head_dim, softmax_scale, workspace, workspace_bytes, status, stream);
}

extern "C" int attn_decode_paged_append(void* out, float* lse, const void* q, void* k_pool, void* v_pool,
                                        const void* k_new, const void* v_new, int num_pages,
                                        const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                                        int batch, int max_seq_len, int page_size, int num_q_heads, int num_kv_heads,
                                        int head_dim, float softmax_scale, void* workspace, size_t workspace_bytes,
                                        int32_t* status, void* stream) {
    NvtxRange nvtx_("attn_decode_paged_append");
    if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return PA_ERR_NULL;
    return dec::launch_decode_kv(out, lse, q, k_pool, v_pool, nullptr, nullptr, k_new, v_new, num_pages, block_table,
                                 max_pages_per_seq, seq_lens, nullptr, batch, 1, 1, batch, max_seq_len, page_size,
                                 num_q_heads, num_kv_heads, head_dim, softmax_scale, workspace, workspace_bytes,
                                 status, stream);
}

extern "C" int attn_decode_multiquery_paged_append(void* out, float* lse, const void* q, void* k_pool, void* v_pool,
                                                   const void* k_new, const void* v_new, int num_pages,
                                                   const int32_t* block_table, int max_pages_per_seq,
                                                   const int32_t* cu_seqlens_q, const int32_t* seq_lens, int batch,
                                                   int total_q, int max_q_len, int max_seq_len, int page_size,
                                                   int num_q_heads, int num_kv_heads, int head_dim,
                                                   float softmax_scale, void* workspace, size_t workspace_bytes,
                                                   int32_t* status, void* stream) {
    NvtxRange nvtx_("attn_decode_multiquery_paged_append");
    if (max_q_len < 1 || max_q_len > kDecodeMaxQ) return PA_ERR_SHAPE;
    if (batch > 0 && (cu_seqlens_q == nullptr || k_new == nullptr || v_new == nullptr)) return PA_ERR_NULL;
    return dec::launch_decode_kv(out, lse, q, k_pool, v_pool, nullptr, nullptr, k_new, v_new, num_pages, block_table,
                                 max_pages_per_seq, seq_lens, cu_seqlens_q, total_q, max_q_len, INT_MAX, batch,
                                 max_seq_len, page_size, num_q_heads, num_kv_heads, head_dim, softmax_scale,
                                 workspace, workspace_bytes, status, stream);
}

extern "C" int attn_decode_multiquery_paged(void* out, float* lse, const void* q, const void* k_pool,
                                            const void* v_pool, int num_pages, const int32_t* block_table,
                                            int max_pages_per_seq, const int32_t* cu_seqlens_q,
                                            const int32_t* seq_lens, int batch, int total_q, int max_q_len,
                                            int max_seq_len, int page_size, int num_q_heads, int num_kv_heads,
                                            int head_dim, float softmax_scale, void* workspace,
                                            size_t workspace_bytes, int32_t* status, void* stream) {
    NvtxRange nvtx_("attn_decode_multiquery_paged");
    if (max_q_len < 1 || max_q_len > kDecodeMaxQ) return PA_ERR_SHAPE;
    if (batch > 0 && cu_seqlens_q == nullptr) return PA_ERR_NULL;
    return dec::launch_decode(out, lse, q, k_pool, v_pool, num_pages, block_table, max_pages_per_seq, seq_lens,
                              cu_seqlens_q, total_q, max_q_len, INT_MAX, batch, max_seq_len, page_size,
                              num_q_heads, num_kv_heads, head_dim, softmax_scale, workspace, workspace_bytes,
                              status, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free decode entry point.
//
// Some callers cannot call cudaMalloc: code running inside an allocator or
// memory-pool callback, a plugin loaded into a host framework that owns all
// device memory, or a latency-critical path that must not enter the driver's
// allocator.  For them this file keeps the split-K scratch (the partial
// outputs) in a fixed device array, so the only buffers they pass are
// inputs and outputs.
// ---------------------------------------------------------------------------
namespace pa {
namespace dec {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB held by every GPU that loads the library

// Zero at module load.  Shared by every call on the device.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_static_mu;
void* g_static_ptr[64] = {};
unsigned long long g_static_ctx[64] = {};  // context the cached address belongs to
}  // namespace

// Device address of g_static_scratch on the current device, looked up once
// per device and context (the host-side name is only a stand-in, not a device
// address).  A context created after a device reset has a new ID, so the
// address is looked up again instead of pointing into the old context's memory.
static int static_scratch_ptr(int device, void** out) {
    if (device < 0 || device >= 64) return PA_ERR_CUDA;
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != PA_OK) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (g_static_ptr[device] == nullptr || g_static_ctx[device] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        g_static_ptr[device] = p;
        g_static_ctx[device] = ctx;
    }
    *out = g_static_ptr[device];
    return PA_OK;
}

}  // namespace dec
}  // namespace pa

extern "C" int attn_decode_paged_noalloc(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                                         int num_pages, const int32_t* block_table, int max_pages_per_seq,
                                         const int32_t* seq_lens, int batch, int max_seq_len, int page_size,
                                         int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                                         int32_t* status, void* stream) {
    NvtxRange nvtx_("attn_decode_paged_noalloc");
    if (batch < 0) return PA_ERR_SHAPE;
    int rc = check_common_shapes(page_size, num_q_heads, num_kv_heads, head_dim);
    if (rc != PA_OK) return rc;
    if (batch == 0) return PA_OK;
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc != PA_OK) return rc;
    const size_t need = pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim);
    if (need == 0) return PA_ERR_SHAPE;
    if (need > dec::kStaticScratchBytes) return PA_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    rc = dec::static_scratch_ptr(dev.device, &scratch);
    if (rc != PA_OK) return rc;
    return attn_decode_paged(out, lse, q, k_pool, v_pool, num_pages, block_table, max_pages_per_seq, seq_lens, batch,
                             max_seq_len, page_size, num_q_heads, num_kv_heads, head_dim, softmax_scale, scratch,
                             dec::kStaticScratchBytes, status, stream);
}
