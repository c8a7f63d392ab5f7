// The mixed serving step in one persistent launch: the split-K decode of the
// short entries (q_len <= 8) and the tcgen05 prefill of the long ones.
//
// What it computes is exactly what the separate kernels compute ("Inside Ion",
// section "IonAttention in One Paragraph": one fused prefill-plus-decode
// attention kernel; chunked prefill next to decode rows as in "The Stack Below
// the Stack, Part 2", closing recipe): decode rows through Flash-Decoding with
// the log-sum-exp merge, prefill tiles through the online-softmax tile loop.
//
// GB300 design
// * One CTA of three warpgroups (384 threads) per SM, persistent.  The two roles
//   want very different register budgets -- the decode's mma.sync pipeline keeps
//   about 240 registers per thread in 4 warps, the prefill's 11 warps fit in 168
//   -- so the budget changes with the phase (setmaxnreg): the launch gives every
//   thread 168, the decode phase moves 144 of warpgroup 2's registers per thread
//   to warpgroups 0 and 1 (240 each, warpgroup 2 at 24), and the prefill phase
//   gives them back.
// * Phase 1, decode: warpgroups 0 and 1 are two "virtual CTAs" of the split-K
//   decode (the decode kernel's body, each with its own half of shared memory and
//   its own named barrier), 2 per SM as in the stand-alone decode grid.  They take
//   equal ranges of the decode work units.  Meanwhile warpgroup 2 of CTA 0 builds
//   the prefill plan -- every query tile of the long entries, sorted by cost,
//   heaviest first -- in the workspace and publishes it with a flag tagged with
//   this launch's grid ID.
// * Phase 2, prefill: the prefill kernel's roles (softmax warps 0-7, producer 8,
//   MMA issuers 9-10) on the same shared memory and tensor memory.  Work items are
//   claimed one at a time by a fetch-and-add on a counter that the plan's builder
//   set up (tagged with the grid ID) before publishing the plan, so a CTA whose
//   decode range ended early takes more of the heaviest-first list: the ragged end
//   of the decode phase fills with prefill work instead of idling.
// * The merge of split decode rows is a second, small kernel launched as this
//   one's programmatic dependent (as after the stand-alone decode).
#include "decode_dev.cuh"
#include "prefill_dev.cuh"
#include "pa_trace.h"

#include <mutex>

namespace pa {
namespace mix {

constexpr int NTHREADS = 384;  // three warpgroups
constexpr int DEC_REGS = 240;  // registers per thread of warpgroups 0 and 1 while they decode
constexpr int IDLE_REGS = 24;  // warpgroup 2 meanwhile (384 * 168 = 2 * 128 * 240 + 128 * 24)
constexpr int PF_REGS = 168;   // every warpgroup in the prefill phase
constexpr int PLAN_BAR = 3;    // named barrier of warpgroup 2 while it builds the plan
static_assert(2 * 128 * DEC_REGS + 128 * IDLE_REGS <= NTHREADS * PF_REGS, "register split over the launch budget");

constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }

template <int D>
struct MCfg {
    using DC = dec::Cfg<D, false, false>;
    using DS = dec::DecShared<D, false, 2>;
    static constexpr int VCTA_BYTES = align1k(DC::STAGES_BYTES + DC::MERGE_BYTES + (int)sizeof(DS));
    static constexpr int DS_OFF = DC::STAGES_BYTES + DC::MERGE_BYTES;  // DecShared inside a virtual CTA's part
    static constexpr int PLAN_OFF = 2 * VCTA_BYTES;                    // warpgroup 2's scan scratch
    static constexpr int DEC_BYTES = PLAN_OFF + 64;
    static constexpr int PF_BYTES = pf::Cfg<D>::SMEM_BYTES - 1024;
    static constexpr int SMEM_BYTES = 1024 + (DEC_BYTES > PF_BYTES ? DEC_BYTES : PF_BYTES);
};

struct MixParams {
    dec::Params d;
    pf::Params f;
    int32_t* hist;  // plan: cost histogram, then running offsets
    int2* tiles;    // plan: the sorted list (f.tiles, writable)
    int32_t* n_tiles;
    unsigned long long* plan_flag;
    unsigned long long* item_ctr;
    int max_cost, cap;
};

template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// This launch's tag: the grid ID (a per-context launch number), never 0 -- the merge
// kernel after the launch resets the plan flag and the item counter to 0.
__device__ __forceinline__ uint32_t grid_tag() {
    uint64_t g;
    asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
    const uint32_t t = (uint32_t)g ^ (uint32_t)(g >> 32);
    return t != 0u ? t : 0x9E3779B9u;
}

__device__ __forceinline__ void plan_sync() {
    asm volatile("bar.sync %0, 128;" ::"n"(PLAN_BAR) : "memory");
}

// Warpgroup 2 of CTA 0: list every 128-row query tile of the entries with
// q_len > kDecodeMaxQ, sorted by the number of 128-key tiles it attends (counting
// sort, heaviest first), then publish the list (flag = grid tag).  t: 0 .. 127.
__device__ __forceinline__ void build_plan(const MixParams& mp, const int t, int* scratch, const uint32_t tag) {
    const pf::Params& f = mp.f;
    for (int c = t; c <= mp.max_cost; c += 128) atomicExch(mp.hist + c, 0);
    plan_sync();
    for (int b = t; b < f.batch; b += 128) {
        int ql, sl;
        const int nt = pf::seq_tiles(f.cu_q, f.seq_lens, b, mp.cap, f.status, ql, sl);
        for (int i = 0; i < nt; ++i) {
            const int rows = min(pf::BM, ql - i * pf::BM);
            const int cost = min(mp.max_cost, (sl - ql + i * pf::BM + rows - 1) / pf::BN + 1);
            atomicAdd(mp.hist + cost, 1);
        }
    }
    plan_sync();
    // exclusive offsets in descending cost order: thread t owns the costs c_hi .. c_lo
    const int per = (mp.max_cost + 1 + 127) / 128;
    const int c_hi = mp.max_cost - t * per;
    const int c_lo = max(0, c_hi - per + 1);
    int sum = 0;
    for (int c = c_hi; c >= c_lo; --c) sum += atomicAdd(mp.hist + c, 0);
    const int incl = warp_incl_scan(sum);
    const int w = t >> 5;
    if ((t & 31) == 31) scratch[w] = incl;
    plan_sync();
    int run = incl - sum;
    for (int i = 0; i < w; ++i) run += scratch[i];
    for (int c = c_hi; c >= c_lo; --c) run += atomicExch(mp.hist + c, run);  // count out, first slot in
    plan_sync();
    const int total = scratch[0] + scratch[1] + scratch[2] + scratch[3];
    for (int b = t; b < f.batch; b += 128) {
        int ql, sl;
        const int nt = pf::seq_tiles(f.cu_q, f.seq_lens, b, mp.cap, nullptr, ql, sl);
        // eight slot claims in flight at a time: each is an L2 round trip, and the other
        // CTAs wait for this list (a sequence's tiles mostly have distinct costs, so distinct counters)
#pragma unroll 8
        for (int i = 0; i < nt; ++i) {
            const int rows = min(pf::BM, ql - i * pf::BM);
            const int cost = min(mp.max_cost, (sl - ql + i * pf::BM + rows - 1) / pf::BN + 1);
            __stcg(mp.tiles + atomicAdd(mp.hist + cost, 1), make_int2(b, i));
        }
    }
    __threadfence();
    plan_sync();
    if (t == 0) {
        __stcg(mp.n_tiles, total);
        __stcg(mp.item_ctr, (unsigned long long)tag << 32);  // claims start at item 0 of this launch
        __threadfence();
        const unsigned long long v = ((unsigned long long)tag << 32) | 1ull;
        asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(mp.plan_flag), "l"(v) : "memory");
    }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    mixed_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                 const MixParams mp) {
    using M = MCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ pf::Shared sh;
    const int wg = threadIdx.x >> 7;
    const uint32_t tag = grid_tag();
    pdl_launch_dependents();  // the merge kernel may be scheduled (it waits for this grid)

    // ---- phase 1: decode (warpgroups 0, 1) and the prefill plan (warpgroup 2 of CTA 0)
    if (wg < 2) {
        regs_inc<DEC_REGS>();
        uint8_t* vs = smem + wg * M::VCTA_BYTES;
        auto& ds = *reinterpret_cast<typename M::DS*>(vs + M::DS_OFF);
        dec::decode_body<D, false, 2, false>(mp.d, 2 * (int)blockIdx.x + wg, 2 * (int)gridDim.x,
                                             (int)threadIdx.x & 127, 1 + wg, vs, ds);
        __syncwarp();
        regs_dec<PF_REGS>();
    } else {
        regs_dec<IDLE_REGS>();
        if (blockIdx.x == 0) build_plan(mp, (int)threadIdx.x - 256, reinterpret_cast<int*>(smem + M::PLAN_OFF), tag);
        __syncwarp();
        regs_inc<PF_REGS>();
    }
    __syncthreads();  // shared memory changes hands
    pdl_wait();       // (returned already in the decode warps) the previous kernel's writes are visible

    // ---- phase 2: prefill, items claimed from the counter
    pf::prefill_body<D>(qmap, kmap, vmap, omap, mp.f, smem, sh, pf::ItemSource{mp.item_ctr, mp.plan_flag, tag});
}

std::mutex g_occ_mu;
int g_occ[64][2] = {};

template <int D>
int resident_ctas(int device) {
    // the occupancy query needs the kernel's dynamic shared-memory limit raised first
    if (set_smem_limit_once((const void*)mixed_kernel<D>, MCfg<D>::SMEM_BYTES, device, D == 128 ? 17 : 18) != PA_OK)
        return 0;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (device < 0 || device >= 64) return 0;
    int& v = g_occ[device][D == 128 ? 1 : 0];
    if (v == 0) {
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mixed_kernel<D>, NTHREADS, MCfg<D>::SMEM_BYTES) !=
                cudaSuccess ||
            per_sm <= 0)
            return 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0) return 0;
        v = per_sm * sms;
    }
    return v;
}

template <int D>
int launch(cudaStream_t st, int device, int ctas, const CUtensorMap& qmap, const CUtensorMap& kmap,
           const CUtensorMap& vmap, const CUtensorMap& omap, const MixParams& mp) {
    if (set_smem_limit_once((const void*)mixed_kernel<D>, MCfg<D>::SMEM_BYTES, device, D == 128 ? 17 : 18) != PA_OK)
        return PA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)MCfg<D>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mixed_kernel<D>, qmap, kmap, vmap, omap, mp) == cudaSuccess ? PA_OK
                                                                                                : PA_ERR_CUDA;
}

}  // namespace mix

namespace pf {

int launch_fused(int head_dim, cudaStream_t st, void* out, float* lse, const void* q, const void* k_pool,
                 const void* v_pool, int num_pages, const int32_t* block_table, int max_pages_per_seq,
                 const int32_t* cu_seqlens_q, const int32_t* seq_lens, int batch, int total_q, int max_seq_len,
                 int page_size, int num_q_heads, int num_kv_heads, float softmax_scale, void* workspace,
                 size_t dec_bytes, int32_t* status, const CUtensorMap& qmap, const CUtensorMap& kmap,
                 const CUtensorMap& vmap, const CUtensorMap& omap, const Params& prm, const PlanArea& plan,
                 int max_cost) {
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != PA_OK) return rc;
    const int ctas = head_dim == 128 ? mix::resident_ctas<128>(dev.device) : mix::resident_ctas<64>(dev.device);
    if (ctas <= 0) return PA_ERR_CUDA;
    // the decode rows: two virtual CTAs per CTA, their operand order chosen per segment
    dec::DecodeLaunch L;
    rc = dec::prepare_decode(&L, out, lse, q, k_pool, v_pool, nullptr, nullptr, nullptr, nullptr, num_pages,
                             block_table, max_pages_per_seq, seq_lens, cu_seqlens_q, total_q, kDecodeMaxQ,
                             kDecodeMaxQ, batch, max_seq_len, page_size, num_q_heads, num_kv_heads, head_dim,
                             softmax_scale, workspace, dec_bytes, status, /*per_segment=*/true, 2 * ctas);
    if (rc != PA_OK) return rc;
    if (L.grid == 0) return PA_OK;
    mix::MixParams mp;
    mp.d = L.prm;
    mp.f = prm;
    mp.hist = plan.hist;
    mp.tiles = plan.tiles;
    mp.n_tiles = plan.n_tiles;
    mp.plan_flag = plan.flag;
    mp.item_ctr = plan.counter;
    mp.max_cost = max_cost;
    mp.cap = max_pages_per_seq * page_size;
    log_config("mixed step in one launch: head_dim %d, %d CTAs x %d threads (1 per SM); phase 1: split-K decode "
               "of the q_len <= %d entries on 2 virtual CTAs per CTA (%d registers, operand order per segment, min "
               "chunk %d units) while one warpgroup builds the prefill plan; phase 2: prefill items claimed "
               "heaviest first; then the merge (grid %lld x %d)",
               head_dim, ctas, mix::NTHREADS, kDecodeMaxQ, mix::DEC_REGS, L.min_chunk, L.segs, L.nrb_max);
    rc = head_dim == 128 ? mix::launch<128>(st, dev.device, ctas, qmap, kmap, vmap, omap, mp)
                         : mix::launch<64>(st, dev.device, ctas, qmap, kmap, vmap, omap, mp);
    if (rc != PA_OK) return rc;
    L.prm.reset_words = plan.flag;  // flag and counter are adjacent: the merge zeroes both
    rc = dec::launch_merge(L, st);
    if (rc != PA_OK) return rc;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pf
}  // namespace pa
