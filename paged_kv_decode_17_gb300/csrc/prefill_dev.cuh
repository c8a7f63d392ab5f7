// Varlen causal prefill over a paged KV cache on tcgen05 tensor cores (device code).
//
// What it computes ("The Stack Below the Stack, Part 2", section 2.1; "8.
// Kernels and Attention Backends", section "Attention is an I/O problem"):
// exact softmax attention, tiled.  Query tiles of 128 rows and key tiles of
// 128 keys stream through on-chip memory; each row carries a running maximum
// and a running sum of exponentials, and the output accumulated so far is
// rescaled when the maximum grows, so the result equals the untiled softmax.
// Row i of a sequence with q_len rows and seq_len keys sits at position
// seq_len - q_len + i and sees keys 0 .. that position.
//
// GB300 design
// * Work item = one 128-row query tile of one sequence for a pair of query
//   heads of one KV head.  The query tiles are listed sorted by their number of
//   key tiles, heaviest first (by a small plan kernel, or inside the mixed-step
//   kernel).  The kernel is persistent, one CTA per SM; items are taken either
//   round-robin or, in the mixed-step kernel, one at a time from a counter.
//   Tensor memory and barriers are set up once per CTA, and the next item's Q
//   and K/V are loaded while the current item finishes.
// * warp 8 (producer): publishes each item through a 2-slot ring in shared
//   memory, loads the two Q tiles by TMA (3-D tensor map over [rows][Hq][D],
//   128-byte swizzle) and gathers K and V tiles: a 128-key tile is eight
//   16-row page blocks found through the block table (entries loaded four
//   tiles ahead), each one 128-byte-swizzled TMA box of 4 KB at head_dim 128
//   (see Cfg::BLK4; a warp issues about one copy per 110 cycles, so fewer,
//   larger boxes move the tile sooner).  K and V tiles have separate rings
//   (1 and 2 stages), so the next K tile loads as soon as the current scores
//   are computed.
// * warps 9 / 10 (MMA, one per head): one thread issues tcgen05.mma:
//   S_h = Q_h K^T into TMEM (fp32, 128 columns) and O_h += P_h V into TMEM
//   (fp32, D columns); the next tile's scores are issued as soon as the
//   softmax has pulled the current ones out of TMEM.
// * warps 0-3 / 4-7 (softmax, head 0 / 1): thread = row = TMEM lane; the
//   whole score row goes to registers, is masked on diagonal tiles, and
//   2^(s * scale * log2 e - m) becomes P (bf16) in shared memory in the
//   swizzled K-major operand layout.  O is rescaled in TMEM only when a row
//   maximum grows by more than TAU = 8 (log2 units): until then the
//   exponentials are taken against the older, smaller maximum, which keeps
//   them <= 2^8 and the result exact, because the final division uses the
//   same reference maximum for numerator and denominator.  At the end of an
//   item they normalise O; a full 128-row tile goes as bf16 into the head's
//   P buffer (free once the last P.V is done), in the swizzled layout of a
//   TMA box, and one thread writes it out with TMA tensor stores, so the
//   warps move on to the next item at once (the next P store waits only for
//   the store to have read the buffer).  A partial tile is stored directly,
//   row by row, since a whole box would overwrite the next sequence's rows.
// * CTA pairs (PAIR, optional): see Cfg.
// Every wait is bounded; a timeout sets a CTA-wide abort flag, records
// PA_ERR_TIMEOUT and all roles fall through to a clean exit.
#pragma once

#include "pa_common.cuh"
#include "pa_host.h"

namespace pa {
namespace pf {

constexpr int BM = 128;      // query rows per tile (= TMEM lanes)
constexpr int BN = 128;      // keys per KV tile
constexpr int UPT = BN / 16; // 16-key page blocks per KV tile
#ifndef PA_PF_NK
#define PA_PF_NK 1
#endif
#ifndef PA_PF_NV
#define PA_PF_NV 2
#endif
// K and V tiles go through separate rings: the next K tile only waits for the
// current scores (S) to be computed, not for the previous P.V to finish.
constexpr int NK = PA_PF_NK;  // K ring depth
constexpr int NV = PA_PF_NV;  // V ring depth
// CTA pairs (cta_group::2, below) stage half tiles, so deeper rings fit
constexpr int PNK = 2, PNV = 3;
constexpr int NSTAGE_MAX = PNK + PNV;  // stages 0 .. NK-1 hold K tiles, the next NV V tiles
constexpr float TAU = 8.f;   // rescale threshold, log2 units
// warps 0-7: softmax (head = warp / 4, row quarter = warp & 3)
// warp 8: producer; warps 9 and 10: MMA issuers of head 0 and head 1
constexpr int NTHREADS = 352;
constexpr int WARP_TMA = 8, WARP_MMA0 = 9;
constexpr int PLAN_THREADS = 512;

// PAIR: a cluster of two CTAs on two SMs runs each tile as one M = 256 MMA
// (cta_group::2): each CTA holds its own 128 query rows (two heads' Q and P), half of
// every K tile (keys 0-63 in the first CTA, 64-127 in the second) and half of every V
// tile (value columns 0-63 / 64-127); the MMA reads the other half from the peer's
// shared memory, and each CTA's tensor memory receives its own rows' S and O.
template <int D, bool PAIR = false>
struct Cfg {
    static_assert(!PAIR || D == 128, "a CTA pair splits V into two 128-byte column blocks");
    static constexpr int KB = D / 64;               // 128-byte column blocks per row
    // BLK4: a 16-key page block (16 rows x 256 bytes, contiguous in the pool) is one TMA box,
    // landing as [row half][column block][8 rows][128 bytes], so a stage holds page block u at
    // u * 4096 and every 8-row swizzle atom of one column block sits 2048 bytes after the last.
    // Otherwise (head_dim 64, CTA pairs) a box is 16 rows of one column block, stages [kb][u].
    static constexpr bool BLK4 = !PAIR && D == 128;
    static constexpr int NKr = PAIR ? PNK : NK;     // ring depths
    static constexpr int NVr = PAIR ? PNV : NV;
    static constexpr int NST = NKr + NVr;
    static constexpr int Q_BYTES = BM * D * 2;      // one head's Q tile
    static constexpr int KV_BYTES = BN * D * 2 / (PAIR ? 2 : 1);  // one K or V stage
    static constexpr int P_BYTES = BM * BN * 2;     // one P tile
    static constexpr int Q_KB = BM * 128;           // bytes per column block of a Q tile
    static constexpr int KV_KB = BN * 128;          // bytes per column block of a V stage (of a K stage, unpaired)
    static constexpr int K_KB = (PAIR ? BN / 2 : BN) * 128;  // bytes per column block of a K stage
    static constexpr int VKB = PAIR ? 1 : KB;       // column blocks per V stage
    static constexpr int P_KB = BM * 128;           // bytes per 64-key column block of a P tile
    static constexpr int OFF_Q = 0;                 // Q[head]
    static constexpr int OFF_P = 2 * Q_BYTES;       // P[head]
    static constexpr int OFF_KV = OFF_P + 2 * P_BYTES;
    static constexpr int SMEM_BYTES = 1024 + OFF_KV + NST * KV_BYTES;
    // TMEM columns: S[head] (BN fp32), O[head] (D fp32)
    static constexpr int TM_S0 = 0;
    static constexpr int TM_O0 = 2 * BN;
    static constexpr int TM_USED = 2 * BN + 2 * D;
    static constexpr int TM_COLS = TM_USED <= 256 ? 256 : 512;
    static_assert(TM_USED <= 512, "more than the 512 TMEM columns");
    static constexpr int MM = PAIR ? 2 * BM : BM;   // rows of one MMA
    static constexpr uint32_t IDESC_S = tc::idesc_bf16(MM, BN, 0, 0);   // Q K-major, K K-major
    static constexpr uint32_t IDESC_PV = tc::idesc_bf16(MM, D, 0, 1);   // P K-major, V MN-major
};

struct Params {
    __nv_bfloat16* out;
    float* lse;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* cu_q;
    const int2* tiles;       // plan: (sequence, query tile) sorted heaviest first
    const int32_t* n_tiles;  // plan: number of entries
    int32_t* status;
    int num_pages, max_pages, batch, page_size;
    int Hq, Hkv, group;
    int NPC;  // head pairs (CTA pairs: blocks of 4 heads) per KV head
    unsigned long long wait_ns;  // limit of any one wait (kWaitTimeoutNs unless overridden for tests)
    float scale_log2;
};

// One work item as published by the producer.
struct Item {
    int end;  // 1: no more items
    int b, t, q_len, seq_len, row0, g, h0, nheads, n_kv, rows_valid, qmin;
    int nstore;  // head slots whose results are stored (a CTA pair computes a last valid head twice)
    int hmax;    // last query head of the KV group: slots past it compute it again
};

struct Shared {
    uint64_t bar_q[2], q_empty[2];  // per head: Q tile landed / Q tile no longer read
    uint64_t kv_full[NSTAGE_MAX];
    uint64_t kv_empty[NSTAGE_MAX];
    uint64_t v_peer[PNV];                // CTA pairs: the second CTA has cleared its rows of a V tile past the end
    uint64_t s_full[2], s_free[2];
    uint64_t p_ready[2], pv_done[2];
    uint64_t o_free[2];                  // per head: the epilogue has read O out of TMEM
    uint64_t o_staged[2];                // per head: all 128 rows of O/l are in shared memory
    uint64_t o_read[2];                  // per head: the TMA store has read them (P buffer free again)
    uint64_t v_tail;                     // TMA copies of a V tile that runs past the sequence end land here
    uint64_t mma_drain;                  // per MMA warp: all of its tensor-core operations have completed
    uint64_t item_full[2], item_empty[2];
    uint32_t tmem_base;
    int abort_flag;
    Item items[2];
};

// ---------------------------------------------------------------------------------- CTA pairs
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_cta(const void* local, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    return a;
}

// Arrive (release, cluster scope) on an mbarrier given by its cluster address.
__device__ __forceinline__ void arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// TMA loads into this CTA's shared memory whose completion is counted on the first
// CTA's barrier (cluster address `bar`).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

namespace tc2 {  // tcgen05 for CTA pairs (a kernel uses one CTA group throughout)
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the barrier at cluster address `bar` once this thread's MMAs are done.
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
}  // namespace tc2

// Bounded wait that reports nothing (drains): true once the phase completed.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 <= limit_ns)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Wait for phase `parity` of `bar`; false (and every other role falls through) once any
// role of the CTA has waited longer than p.wait_ns, which records PA_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, Shared& sh, const Params& p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(&sh.abort_flag)) return false;
        if (globaltimer_ns() - t0 > p.wait_ns) {
            *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
            report(p.status, PA_ERR_TIMEOUT);
            return false;
        }
    }
}

// One 16-key page block of a pool (5-D map: 64 columns, 8 rows, column block, row half,
// 16-row block of the pool); the other coordinates are 0.
__device__ __forceinline__ void tma_load_block(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int blk) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %3, %3, %3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(0), "r"(blk)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// 32 lanes x 8 columns of 32-bit: thread t of the warp loads / stores its lane's 8 columns.
__device__ __forceinline__ void ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float m;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
    return m;
}

// (d0, d1) = (x0, x1) * s + (c, c), one packed FFMA (each lane rounded as fmaf)
__device__ __forceinline__ void ffma2(float& d0, float& d1, float x0, float x1, float s, float c) {
    uint64_t x, sv, cv, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(sv) : "f"(s));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cv) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(sv), "l"(cv));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}

// (a0, a1) += (b0, b1), one packed add
__device__ __forceinline__ void fadd2(float& a0, float& a1, float b0, float b1) {
    uint64_t a, b, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(d));
}

// TMA tensor store of one 64-column x 128-row box of O (3-D map over out [rows][Hq][D]).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// number of 128-row query tiles of sequence b served by the prefill kernel (0 if none)
__device__ __forceinline__ int seq_tiles(const int32_t* cu_q, const int32_t* seq_lens, int b, int cap,
                                         int32_t* status, int& q_len, int& seq_len) {
    q_len = __ldg(cu_q + b + 1) - __ldg(cu_q + b);
    seq_len = __ldg(seq_lens + b);
    if (q_len < 0 || seq_len < q_len || seq_len > cap) {
        report(status, PA_ERR_BAD_LEN);
        return 0;
    }
    if (q_len <= kDecodeMaxQ) return 0;  // short query blocks go to the split-K decode kernel
    return (q_len + BM - 1) / BM;
}

// ---------------------------------------------------------------------------------- items
// Where the producer finds this CTA's k-th work item.  Without a counter: the static
// round-robin walk blockIdx.x + k * gridDim.x of the sorted list (head slots rotated by
// the tile index).  With one: the next
// unclaimed item, one fetch-and-add on a 64-bit counter, so CTAs that finish earlier
// work take more items.  The plan is then built inside the same launch: whoever builds
// it sets the counter to (tag << 32) before it publishes plan_flag = (tag << 32) | 1,
// and a producer claims only after it has seen that flag.  (A compare-and-swap loop
// that restarted stale counts itself serialised the 152 producers: 1.9x slower.)
struct ItemSource {
    unsigned long long* counter;
    const unsigned long long* plan_flag;
    uint32_t tag;
};

// Next item index, or -1 if the counter does not belong to this launch.
__device__ __forceinline__ long long claim_item(unsigned long long* ctr, uint32_t tag) {
    const unsigned long long old = atomicAdd(ctr, 1ull);
    return (uint32_t)(old >> 32) == tag ? (long long)(old & 0xffffffffull) : -1;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* a) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}

// ---------------------------------------------------------------------------------- main
// One persistent CTA's prefill work: warps 0-7 softmax, 8 producer, 9-10 MMA; any
// further warps only take part in the CTA-wide barriers.  smem: 1024-byte aligned,
// Cfg<D>::SMEM_BYTES - 1024 bytes.
template <int D, bool PAIR = false>
__device__ __forceinline__ void prefill_body(const CUtensorMap& qmap, const CUtensorMap& kmap,
                                             const CUtensorMap& vmap, const CUtensorMap& omap, const Params& p,
                                             uint8_t* smem, Shared& sh, const ItemSource src) {
    using C = Cfg<D, PAIR>;
    constexpr int NKr = C::NKr, NVr = C::NVr;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = PAIR ? cluster_rank() : 0u;  // 0: the CTA that issues the pair's MMAs
    const bool lead = crank == 0;
    // per-warp arrivals of the softmax warps (of both CTAs of a pair) on the MMA-side barriers
    constexpr int SMX_ARRIVALS = PAIR ? 8 : 4;

    if (tid == 0) {
        sh.abort_flag = 0;
        for (int h = 0; h < 2; ++h) {
            mbar_init(&sh.bar_q[h], 1);
            mbar_init(&sh.q_empty[h], 1);
            mbar_init(&sh.s_full[h], 1);
            mbar_init(&sh.s_free[h], SMX_ARRIVALS);
            mbar_init(&sh.p_ready[h], SMX_ARRIVALS);
            mbar_init(&sh.pv_done[h], 1);
            mbar_init(&sh.o_free[h], SMX_ARRIVALS);
            mbar_init(&sh.o_staged[h], 4 * 32);
            mbar_init(&sh.o_read[h], 1);
            mbar_init(&sh.item_full[h], 1);
            mbar_init(&sh.item_empty[h], 2 + 8);  // lane 0 of both MMA warps and of the 8 softmax warps
        }
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&sh.kv_full[s], 1);   // the (first CTA's) producer arms it for the whole tile
            mbar_init(&sh.kv_empty[s], 2);  // released by both MMA threads
        }
        for (int s = 0; s < PNV; ++s) mbar_init(&sh.v_peer[s], 1);
        mbar_init(&sh.v_tail, 1);
        mbar_init(&sh.mma_drain, 2);
        fence_mbar_init();
    }
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs' barriers exist before either signals the other's
    if (warp == WARP_TMA) {
        if (PAIR) {
            tc2::tmem_alloc(&sh.tmem_base, C::TM_COLS);
            tc2::tmem_relinquish();
        } else {
            tc::tmem_alloc(&sh.tmem_base, C::TM_COLS);
            tc::tmem_relinquish();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh.tmem_base;

    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sP = smem + C::OFF_P;
    uint8_t* sKV = smem + C::OFF_KV;

    if (warp == WARP_TMA) {
        // ===================================================== producer (whole warp)
        if (lane == 0) {
            prefetch_tensormap(&qmap);
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
        bool ok = true;
        if (src.plan_flag != nullptr) {  // the list is built in this launch: wait until it is published
            bool ready = false;
            if (lane == 0) {
                const uint64_t t0 = globaltimer_ns();
                while (!(ready = (uint32_t)(ld_acquire_u64(src.plan_flag) >> 32) == src.tag)) {
                    if (globaltimer_ns() - t0 > p.wait_ns) {
                        *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
                        report(p.status, PA_ERR_TIMEOUT);
                        break;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ready, 0);
        }
        const long long n_items = ok ? (long long)(*reinterpret_cast<const volatile int32_t*>(p.n_tiles)) * p.Hkv * p.NPC : 0;
        int kring = 0, vring = 0;     // K / V tiles issued so far
        int tails = 0;                // v_tail phases waited for
        int tails_armed = 0;          // v_tail phases armed (copies issued)
        bool v_open[NVr] = {};        // V stage armed through v_tail, its kv_full arrival not yet made
        int qloads[2] = {0, 0};       // Q tiles loaded per head
        for (int k = 0; ok; ++k) {
            // ---- next item of this CTA (of this pair: both CTAs walk the same list)
            long long it = PAIR ? (long long)(blockIdx.x >> 1) + (long long)k * (gridDim.x >> 1)
                                : (long long)blockIdx.x + (long long)k * gridDim.x;
            if (src.counter != nullptr) {
                long long c = n_items;
                if (lane == 0 && ok) {
                    c = claim_item(src.counter, src.tag);
                    if (c < 0) {  // not set up by this launch: report and stop taking items
                        report(p.status, PA_ERR_TIMEOUT);
                        c = n_items;
                    }
                }
                it = __shfl_sync(0xffffffffu, c, 0);
            }
            Item itm;
            itm.end = it >= n_items;
            if (!itm.end) {
                const int per = p.Hkv * p.NPC;
                const int ti = (int)(it / per);
                int rem = (int)(it - (long long)ti * per);
                // the static round-robin (no counter) hands a CTA every gridDim-th item; with
                // gridDim a multiple of per, it would always draw the same head slot, so the
                // CTAs drawing a group's lone last head would idle at the end: rotate the slots
                // by the tile index (a permutation within each tile)
                if (src.counter == nullptr) rem = (rem + ti) % per;
                itm.g = rem / p.NPC;
                const int pair = rem - itm.g * p.NPC;  // (CTA pairs: block of 4 heads)
                const int2 bt = __ldcg(p.tiles + ti);
                itm.b = bt.x;
                itm.t = bt.y;
                const int c0 = __ldg(p.cu_q + itm.b);
                itm.q_len = __ldg(p.cu_q + itm.b + 1) - c0;
                itm.seq_len = __ldg(p.seq_lens + itm.b);
                itm.row0 = c0 + itm.t * BM;
                const int hfirst = PAIR ? 4 * pair + 2 * (int)crank : 2 * pair;  // within the KV group
                itm.h0 = itm.g * p.group + hfirst;
                itm.nstore = max(0, min(2, p.group - hfirst));
                itm.nheads = PAIR ? 2 : itm.nstore;  // a pair computes both slots (the MMA spans both CTAs)
                itm.hmax = itm.g * p.group + p.group - 1;
                itm.rows_valid = min(BM, itm.q_len - itm.t * BM);
                itm.qmin = itm.seq_len - itm.q_len + itm.t * BM;
                itm.n_kv = (itm.qmin + itm.rows_valid - 1) / BN + 1;
            }
            // block-table entries of four key tiles at a time, one per lane (tile t0 + lane / 8,
            // page block lane % 8), loaded four tiles before they are used, so the table's
            // latency hides behind the copies; the first four load while this item is published
            const int32_t* btab = itm.end ? p.block_table : p.block_table + (size_t)itm.b * p.max_pages;
            auto fetch4 = [&](int t0) -> int {
                const int key0 = (t0 + (lane >> 3)) * BN + (lane & 7) * 16;
                return (!itm.end && key0 < itm.seq_len) ? __ldg(btab + key0 / p.page_size) : -1;
            };
            int ent_next = fetch4(0);
            const int slot = k & 1;
            ok = __all_sync(0xffffffffu, wait_ab(&sh.item_empty[slot], ((k >> 1) & 1) ^ 1, sh, p));
            if (!ok) break;
            if (lane == 0) {
                sh.items[slot] = itm;
                mbar_arrive(&sh.item_full[slot]);  // release: the item is visible to whoever waits
            }
            if (itm.end) break;

            // ---- Q tiles of this item (a head's Q buffer is free once its last S MMA is done)
            for (int hh = 0; hh < itm.nheads && ok; ++hh) {
                if (qloads[hh] > 0)
                    ok = __all_sync(0xffffffffu,
                                    wait_ab(&sh.q_empty[hh], (qloads[hh] - 1) & 1, sh, p));
                if (!ok) break;
                if (lane == 0) {
                    const int head = min(itm.h0 + hh, itm.hmax);
                    if (!PAIR) {
                        mbar_arrive_expect_tx(&sh.bar_q[hh], C::Q_BYTES);
                        for (int kb = 0; kb < C::KB; ++kb)
                            tma_load_3d(sQ + hh * C::Q_BYTES + kb * C::Q_KB, &qmap, &sh.bar_q[hh], kb * 64, head,
                                        itm.row0);
                    } else {
                        // both CTAs' Q tiles land on the first CTA's barrier, armed there for both
                        if (lead) mbar_arrive_expect_tx(&sh.bar_q[hh], 2 * C::Q_BYTES);
                        const uint32_t bq = map_cta(&sh.bar_q[hh], 0);
                        for (int kb = 0; kb < C::KB; ++kb)
                            tma_load_3d_pair(sQ + hh * C::Q_BYTES + kb * C::Q_KB, &qmap, bq, kb * 64, head,
                                             itm.row0);
                    }
                }
                ++qloads[hh];
            }
            if (!ok) break;

            // ---- K / V tiles.  A tile is UPT x KB boxes: 16-key page blocks x 64-column halves
            // (one box per block at head_dim 128).  Lane u < UPT holds the pool row of block u.
            int ent = -1;
            for (int j = 0; j < itm.n_kv && ok; ++j) {
                if ((j & 3) == 0) {
                    ent = ent_next;
                    ent_next = fetch4(j + 4);
                }
                const int phys = __shfl_sync(0xffffffffu, ent, ((j & 3) << 3) + (lane & 7));
                int my_row = -1;  // pool row of block `lane` of tile j, -1 if none
                if (lane < UPT) {
                    const int key0 = j * BN + lane * 16;
                    if (key0 < itm.seq_len) {
                        if (phys < 0 || phys >= p.num_pages)
                            report(p.status, PA_ERR_BAD_PAGE);
                        else
                            my_row = (phys * p.Hkv + itm.g) * p.page_size + key0 % p.page_size;
                    }
                }
                const unsigned goodmask = __ballot_sync(0xffffffffu, my_row >= 0) & ((1u << UPT) - 1);
                const int good = __popc(goodmask);
                const bool tail = (j + 1) * BN > itm.seq_len;
                for (int x = 0; x < 2 && ok; ++x) {
                    const int i = x == 0 ? kring : vring;
                    const int depth = x == 0 ? NKr : NVr;
                    const int st = (x == 0 ? 0 : NKr) + i % depth;
                    ok = __all_sync(0xffffffffu,
                                    wait_ab(&sh.kv_empty[st], ((i / depth) & 1) ^ 1, sh, p));
                    if (!ok) break;
                    if (x == 0)
                        ++kring;  // counted once armed: the drain below waits for armed tiles only
                    else
                        ++vring;
                    uint8_t* dst = sKV + st * C::KV_BYTES;
                    // this lane's box: page block u, 64-column block kb, and its place in the stage.
                    // Unpaired: all UPT x KB boxes.  Pair: K keys 64 r .. 64 r + 63 (blocks 4 r .. 4 r + 3,
                    // both column blocks), V columns 64 r .. 64 r + 63 of every block.
                    int u, kb, off;
                    bool has;
                    if (C::BLK4) {
                        u = lane;
                        kb = 0;
                        has = lane < UPT;
                        off = u * 4096;
                    } else if (!PAIR) {
                        u = lane / C::KB;
                        kb = lane - u * C::KB;
                        has = lane < UPT * C::KB;
                        off = kb * C::KV_KB + u * 2048;
                    } else if (x == 0) {
                        u = 4 * (int)crank + (lane >> 1);
                        kb = lane & 1;
                        has = lane < 8;
                        off = kb * C::K_KB + (lane >> 1) * 2048;
                    } else {
                        u = lane;
                        kb = (int)crank;
                        has = lane < UPT;
                        off = u * 2048;
                    }
                    const int box_row = __shfl_sync(0xffffffffu, my_row, u & 31);
                    const bool mine = has && box_row >= 0;
                    const bool via_tail = (x == 1) && tail;
                    const CUtensorMap* map = x == 0 ? &kmap : &vmap;
                    if (!via_tail) {
                        if (lane == 0 && lead) {  // armed for the whole tile (both CTAs of a pair)
                            if (good == 0)
                                mbar_arrive(&sh.kv_full[st]);
                            else
                                mbar_arrive_expect_tx(&sh.kv_full[st], good * 16 * D * 2);
                        }
                        __syncwarp();
                        if (mine) {
                            if (PAIR)
                                tma_load_2d_pair(dst + off, map, map_cta(&sh.kv_full[st], 0), kb * 64, box_row);
                            else if (C::BLK4)
                                tma_load_block(dst + off, map, &sh.kv_full[st], box_row >> 4);
                            else
                                tma_load_2d(dst + off, map, &sh.kv_full[st], kb * 64, box_row);
                        }
                    } else {
                        // keys past the sequence end: their V rows may hold anything and 0 * NaN = NaN,
                        // so this CTA's copies land on v_tail and it zeroes those rows of its columns
                        // before it lets any MMA read the tile
                        const int own_bytes = good * 16 * 128 * C::VKB;
                        if (lane == 0) {
                            if (own_bytes == 0)
                                mbar_arrive(&sh.v_tail);
                            else
                                mbar_arrive_expect_tx(&sh.v_tail, own_bytes);
                        }
                        __syncwarp();
                        if (mine) {
                            if (C::BLK4)
                                tma_load_block(dst + off, map, &sh.v_tail, box_row >> 4);
                            else
                                tma_load_2d(dst + off, map, &sh.v_tail, kb * 64, box_row);
                        }
                        ++tails_armed;
                        v_open[st - NKr] = true;
                        ok = __all_sync(0xffffffffu, wait_ab(&sh.v_tail, tails & 1, sh, p));
                        if (!ok) break;
                        ++tails;
                        const int first = itm.seq_len - j * BN;
                        const int nchunk = (BN - first) * 8 * C::VKB;  // 16-byte chunks to clear
                        for (int c = lane; c < nchunk; c += 32) {
                            const int cb = c / ((BN - first) * 8);
                            const int rem = c - cb * (BN - first) * 8;
                            const int r = first + rem / 8;
                            const int roff = C::BLK4 ? (r >> 4) * 4096 + ((r >> 3) & 1) * 2048 + cb * 1024 + (r & 7) * 128
                                                     : cb * C::KV_KB + r * 128;
                            *reinterpret_cast<uint4*>(dst + roff + (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (lead)
                                mbar_arrive(&sh.kv_full[st]);
                            else
                                arrive_cluster(map_cta(&sh.v_peer[st - NKr], 0));
                        }
                        v_open[st - NKr] = false;
                    }
                }
            }
        }
        // Before leaving (also after an abort): every TMA copy issued into this CTA has
        // landed.  Older tiles of a stage were consumed before the stage was re-armed, so
        // only the last tile of each stage can still be in flight; a V tile armed through
        // v_tail whose kv_full arrival was never made lands on v_tail.  In a pair the
        // second CTA's copies land on the first CTA's barriers: the first CTA waits for
        // what it armed (after an abort a phase may lack copies the peer never issued,
        // hence the short limit), and copies the peer issued for a phase the first CTA
        // never armed are covered at the very end (both CTAs wait out any copy in flight
        // when either of them aborted).
        if (lane == 0) {
            if (lead) {
                const uint64_t lim = PAIR ? 5000000ull : kWaitTimeoutNs;
                for (int hh = 0; hh < 2; ++hh)
                    if (qloads[hh] > 0) mbar_wait_for(&sh.bar_q[hh], (qloads[hh] - 1) & 1, lim);
                for (int i = max(0, kring - NKr); i < kring; ++i)
                    mbar_wait_for(&sh.kv_full[i % NKr], (i / NKr) & 1, lim);
                for (int i = max(0, vring - NVr); i < vring; ++i)
                    if (!v_open[i % NVr]) mbar_wait_for(&sh.kv_full[NKr + i % NVr], (i / NVr) & 1, lim);
            }
            if (tails_armed > tails) mbar_wait(&sh.v_tail, (tails_armed - 1) & 1);
        }
        __syncwarp();
    } else if (warp == WARP_MMA0 || warp == WARP_MMA0 + 1) {
        // ===================================================== MMA issuer of one head
        const int hh = warp - WARP_MMA0;
        if (PAIR && !lead) {
            // the second CTA of a pair issues no MMA (the first CTA's M = 256 MMAs cover its rows):
            // it only follows the item ring
            if (lane == 0)
                for (int k = 0;; ++k) {
                    if (!wait_ab(&sh.item_full[k & 1], (k >> 1) & 1, sh, p)) break;
                    const bool end = sh.items[k & 1].end != 0;
                    mbar_arrive(&sh.item_empty[k & 1]);
                    if (end) break;
                }
        } else if (lane == 0) {
            const uint32_t qaddr = smem_u32(sQ) + hh * C::Q_BYTES;
            const uint32_t paddr = smem_u32(sP) + hh * C::P_BYTES;
            const uint32_t kv_base = smem_u32(sKV);
            const uint32_t t_s = tmem + C::TM_S0 + hh * BN;
            const uint32_t t_o = tmem + C::TM_O0 + hh * D;
            // completion of this thread's MMAs signalled on a barrier (of both CTAs of a pair)
            auto commit_to = [&](uint64_t* bar) {
                if (PAIR) {
                    tc2::commit(map_cta(bar, 0));
                    tc2::commit(map_cta(bar, 1));
                } else {
                    tc::commit(bar);
                }
            };
            auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
                if (PAIR)
                    tc2::mma_ss(d, a, b, idesc, acc);
                else
                    tc::mma_ss(d, a, b, idesc, acc);
            };
            // a K/V stage is free once both MMA threads are done with it
            auto release = [&](uint64_t* bar) { commit_to(bar); };
            int kr = 0, vr = 0;  // K / V ring positions (same walk as the producer)
            int vtails[PNV] = {};  // pair: V tiles past the end seen per stage (phases of v_peer)
            // stage and phase of the K / V tile of key tile j of the current item
            auto kst = [&](int j) { return (kr + j) % NKr; };
            auto kph = [&](int j) { return (uint32_t)(((kr + j) / NKr) & 1); };
            auto vst = [&](int j) { return NKr + (vr + j) % NVr; };
            auto vph = [&](int j) { return (uint32_t)(((vr + j) / NVr) & 1); };
            int J = 0;      // tiles this head has computed (phase counter of its S / P barriers)
            int items = 0;  // items this head has computed
            int qn = 0;     // Q tiles consumed
            bool ok = true;
            for (int k = 0; ok; ++k) {
                ok = wait_ab(&sh.item_full[k & 1], (k >> 1) & 1, sh, p);
                if (!ok) break;
                const Item itm = sh.items[k & 1];
                if (itm.end) break;
                const int n = itm.n_kv;
                if (hh >= itm.nheads) {
                    // not our head this time: still release every stage we pass
                    for (int j = 0; j < n && ok; ++j) {
                        ok = wait_ab(&sh.kv_full[kst(j)], kph(j), sh, p);
                        if (ok) release(&sh.kv_empty[kst(j)]);
                        if (ok) ok = wait_ab(&sh.kv_full[vst(j)], vph(j), sh, p);
                        if (ok) release(&sh.kv_empty[vst(j)]);
                    }
                } else {
                    ok = wait_ab(&sh.bar_q[hh], qn & 1, sh, p);
                    ++qn;
                    auto issue_s = [&](int j) {
                        const uint32_t kaddr = kv_base + kst(j) * C::KV_BYTES;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t ad =
                                tc::smem_desc_sw128(qaddr + (kk >> 2) * C::Q_KB + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd =
                                C::BLK4 ? tc::smem_desc_sw128(kaddr + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048)
                                        : tc::smem_desc_sw128(kaddr + (kk >> 2) * C::K_KB + (kk & 3) * 32, 16, 1024);
                            mma(t_s, ad, bd, C::IDESC_S, kk > 0);
                        }
                        commit_to(&sh.s_full[hh]);
                        if (j == n - 1) commit_to(&sh.q_empty[hh]);  // last read of this Q tile
                    };
                    auto issue_pv = [&](int j) {
                        const uint32_t vaddr = kv_base + vst(j) * C::KV_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            const uint64_t ad =
                                tc::smem_desc_sw128(paddr + (kk >> 2) * C::P_KB + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd = C::BLK4 ? tc::smem_desc_sw128(vaddr + kk * 4096, 1024, 2048)
                                                        : tc::smem_desc_sw128(vaddr + kk * 2048, C::KV_KB, 1024);
                            mma(t_o, ad, bd, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        commit_to(&sh.pv_done[hh]);
                    };
                    // scores of key tile 0 (the S buffer was freed by the previous tile's softmax)
                    if (ok) ok = wait_ab(&sh.kv_full[kst(0)], kph(0), sh, p);
                    if (ok && J > 0) ok = wait_ab(&sh.s_free[hh], (J - 1) & 1, sh, p);
                    if (ok) {
                        tc::fence_after_sync();
                        issue_s(0);
                        release(&sh.kv_empty[kst(0)]);
                    }
                    for (int j = 0; j < n && ok; ++j) {
                        if (j + 1 < n) {
                            // next scores as soon as the softmax has pulled the current ones out of TMEM
                            ok = wait_ab(&sh.kv_full[kst(j + 1)], kph(j + 1), sh, p) &&
                                 wait_ab(&sh.s_free[hh], (J + j) & 1, sh, p);
                            if (!ok) break;
                            tc::fence_after_sync();
                            issue_s(j + 1);
                            release(&sh.kv_empty[kst(j + 1)]);
                        }
                        ok = wait_ab(&sh.kv_full[vst(j)], vph(j), sh, p) &&
                             wait_ab(&sh.p_ready[hh], (J + j) & 1, sh, p);
                        if (PAIR && ok && (j + 1) * BN > itm.seq_len) {  // the peer zeroed its rows past the end
                            const int vs = vst(j) - NKr;
                            ok = wait_ab(&sh.v_peer[vs], vtails[vs] & 1, sh, p);
                            ++vtails[vs];
                        }
                        // the first P.V overwrites O: the previous item's epilogue must have read it
                        if (ok && j == 0 && items > 0) ok = wait_ab(&sh.o_free[hh], (items - 1) & 1, sh, p);
                        if (!ok) break;
                        tc::fence_after_sync();
                        issue_pv(j);
                        release(&sh.kv_empty[vst(j)]);
                    }
                    J += n;
                    ++items;
                }
                kr += n;
                vr += n;
                mbar_arrive(&sh.item_empty[k & 1]);
            }
            // every tensor-core operation this thread issued has completed (after an abort some
            // may still run) before the CTA frees tensor memory and leaves
            if (PAIR)
                tc2::commit(map_cta(&sh.mma_drain, 0));
            else
                tc::commit(&sh.mma_drain);
            mbar_wait(&sh.mma_drain, 0);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ===================================================== softmax (thread = row, all BN columns)
        const int hh = warp >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // tile row = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + lane_off + C::TM_S0 + hh * BN;
        const uint32_t t_o = tmem + lane_off + C::TM_O0 + hh * D;
        uint8_t* prow = sP + hh * C::P_BYTES + r * 128;
        // one arrival per warp (after every lane's accesses) on a barrier of the MMA side:
        // in a pair, the first CTA's barrier counts both CTAs' warps
        auto smx_arrive = [&](uint64_t* bar) {
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    arrive_cluster(map_cta(bar, 0));
                else
                    mbar_arrive(bar);
            }
        };
        const bool leader = quarter == 0 && lane == 0;
        int J = 0;  // tiles of this head so far (phase counter, shared with the MMA thread)
        int nst = 0;               // O tiles written out through the P buffer by TMA stores
        bool store_pending = false;  // the last of them may still be reading the P buffer
        bool ok = true;
        for (int k = 0; ok; ++k) {
            ok = __all_sync(0xffffffffu, wait_ab(&sh.item_full[k & 1], (k >> 1) & 1, sh, p));
            if (!ok) break;
            const Item itm = sh.items[k & 1];
            if (itm.end) break;
            if (hh < itm.nheads) {
                const int n = itm.n_kv;
                const int qpos = itm.qmin + r;
                float m_ref = -INFINITY, l = 0.f;
                for (int j = 0; j < n && ok; ++j) {
                    const int jj = J + j;
                    ok = __all_sync(0xffffffffu, wait_ab(&sh.s_full[hh], jj & 1, sh, p));
                    if (!ok) break;
                    tc::fence_after_sync();
                    // the whole score row into registers, then S is free for the next tile's MMA
                    float x[BN];
#pragma unroll
                    for (int c0 = 0; c0 < BN; c0 += 32) {
                        uint32_t sr[32];
                        tc::ld_32x32b_x32(t_s + c0, sr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[c0 + i] = __uint_as_float(sr[i]);
                    }
                    tc::wait_ld();
                    tc::fence_before_sync();
                    smx_arrive(&sh.s_free[hh]);
                    if ((j + 1) * BN - 1 > itm.qmin) {  // diagonal tile: some key is after some row
#pragma unroll
                        for (int c = 0; c < BN; ++c)
                            if (j * BN + c > qpos) x[c] = -INFINITY;
                    }
                    // row max of the raw scores (softmax_scale > 0): eight chains of 3-input maxima
                    float t8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) t8[i] = fmaxf(x[i], x[8 + i]);
#pragma unroll
                    for (int c = 16; c < BN; c += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) t8[i] = fmax3(t8[i], x[c + i], x[c + 8 + i]);
                    const float mx = fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]),
                                           fmaxf(t8[6], t8[7])) *
                                     p.scale_log2;
                    if (j == 0) {
                        m_ref = mx;
                    } else if (__any_sync(0xffffffffu, mx > m_ref + TAU)) {
                        // rescale O to a new reference maximum (all earlier PVs done once PV(j-1) is)
                        const float m_new = fmaxf(m_ref, mx);
                        const float alpha = ex2(m_ref - m_new);
                        ok = __all_sync(0xffffffffu, wait_ab(&sh.pv_done[hh], (jj - 1) & 1, sh, p));
                        if (!ok) break;
                        tc::fence_after_sync();
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 8) {  // 8 columns at a time: the score row stays live
                            uint32_t o[8];
                            ld_32x32b_x8(t_o + c0, o);
                            tc::wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            st_32x32b_x8(t_o + c0, o);
                        }
                        tc::wait_st();
                        l *= alpha;
                        m_ref = m_new;
                    }
                    // p = 2^(s * scale_log2 - m_ref): the arguments two at a time (packed FFMA), one
                    // MUFU each, packed to bf16 in registers while the previous tile's P.V may still
                    // be running; the sum in four packed accumulators
                    const float neg = -m_ref;
                    float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    uint32_t pk[BN / 2];
#pragma unroll
                    for (int q = 0; q < BN / 8; ++q) {  // 16-byte chunk q = keys 8q .. 8q+7
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float a0, a1;
                            ffma2(a0, a1, x[8 * q + 2 * i], x[8 * q + 2 * i + 1], p.scale_log2, neg);
                            const float p0 = ex2(a0), p1 = ex2(a1);
                            fadd2(s8[2 * i], s8[2 * i + 1], p0, p1);
                            pk[4 * q + i] = pack_bf16x2(p0, p1);
                        }
                    }
                    // the P buffer was last read by the previous tile's P.V (possibly of the
                    // previous item).  Waiting for it also keeps p_ready / pv_done within one
                    // phase of their waiters (mbarrier parity only tells adjacent phases apart).
                    if (jj > 0) {
                        ok = __all_sync(0xffffffffu, wait_ab(&sh.pv_done[hh], (jj - 1) & 1, sh, p));
                        if (!ok) break;
                    }
                    // the previous item's O may still be leaving the P buffer through a TMA store
                    if (store_pending) {
                        if (leader) {
                            bulk_wait_read_all();
                            mbar_arrive(&sh.o_read[hh]);
                        }
                        ok = __all_sync(0xffffffffu, wait_ab(&sh.o_read[hh], (nst - 1) & 1, sh, p));
                        if (!ok) break;
                        store_pending = false;
                    }
                    // P (bf16) to shared memory in the 128-byte-swizzled K-major layout
#pragma unroll
                    for (int q = 0; q < BN / 8; ++q) {
                        const int kb = q >> 3, c = q & 7;
                        *reinterpret_cast<uint4*>(prow + kb * C::P_KB + ((c ^ (r & 7)) << 4)) =
                            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                    }
                    l += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
                    fence_proxy_async_smem();
                    tc::fence_before_sync();
                    smx_arrive(&sh.p_ready[hh]);
                }
                // ---- epilogue: O / l -> bf16, then hand O back to the MMA thread
                if (ok)
                    ok = __all_sync(0xffffffffu, wait_ab(&sh.pv_done[hh], (J + n - 1) & 1, sh, p));
                if (ok) {
                    tc::fence_after_sync();
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    // a pair may compute the KV group's last head in two slots: one copy is stored
                    const bool keep = hh < itm.nstore;
                    const bool store = keep && r < itm.rows_valid;
                    const int h = min(itm.h0 + hh, itm.hmax);
                    if (!keep) {
                    } else if (itm.rows_valid == BM) {
                        // full tile: O/l -> bf16 into the P buffer (free: the last P.V is done) in the
                        // swizzled layout of a 64-column TMA box, then one thread stores it with TMA
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t o[32];
                            tc::ld_32x32b_x32(t_o + c0, o);
                            tc::wait_ld();
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint32_t pkd[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    pkd[e] = pack_bf16x2(__uint_as_float(o[8 * i + 2 * e]) * inv,
                                                         __uint_as_float(o[8 * i + 2 * e + 1]) * inv);
                                const int c = ((c0 & 63) >> 3) + i;  // 16-byte chunk within the 64-column block
                                *reinterpret_cast<uint4*>(prow + (c0 >> 6) * C::P_KB + ((c ^ (r & 7)) << 4)) =
                                    make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
                            }
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(&sh.o_staged[hh]);
                        if (leader) {
                            ok = wait_ab(&sh.o_staged[hh], nst & 1, sh, p);
                            if (ok) {
#pragma unroll
                                for (int kb = 0; kb < C::KB; ++kb)
                                    tma_store_3d(&omap, sP + hh * C::P_BYTES + kb * C::P_KB, kb * 64, h, itm.row0);
                                bulk_commit();
                            }
                        }
                        ++nst;
                        store_pending = true;
                    } else {
                    __nv_bfloat16* orow = p.out + ((size_t)(itm.row0 + r) * p.Hq + h) * D;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tc::ld_32x32b_x32(t_o + c0, o);
                        tc::wait_ld();
                        if (store) {
                            uint32_t pkd[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pkd[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv,
                                                     __uint_as_float(o[2 * i + 1]) * inv);
                            uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
                        }
                    }
                    }
                    if (store && p.lse != nullptr)
                        p.lse[(size_t)(itm.row0 + r) * p.Hq + h] = l > 0.f ? (m_ref + lg2(l)) * kLn2 : -INFINITY;
                    tc::fence_before_sync();
                    smx_arrive(&sh.o_free[hh]);
                }
                J += n;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.item_empty[k & 1]);
        }
        if (leader && nst > 0) bulk_wait_all();  // the shared-memory source must outlive the stores
    }

    tc::fence_before_sync();
    __syncthreads();
    if (PAIR) {
        cluster_sync();  // every role of both CTAs is done
        if (tid == 0) {
            // after an abort in either CTA, a TMA copy may still be landing in this CTA's shared
            // memory (issued for a phase the first CTA never armed): wait it out
            uint32_t peer_abort;
            asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(peer_abort) : "r"(map_cta(&sh.abort_flag, crank ^ 1u)));
            if (peer_abort != 0 || *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        }
        cluster_sync();  // neither CTA leaves while the other may still read its flag
    }
    tc::fence_after_sync();
    if (warp == WARP_TMA) {
        if (PAIR)
            tc2::tmem_dealloc(tmem, C::TM_COLS);
        else
            tc::tmem_dealloc(tmem, C::TM_COLS);
    }
}

// PAIR: launched in clusters of two CTAs (the pair), gridDim.x even.
template <int D, bool PAIR>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                   const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Shared sh;
    prefill_body<D, PAIR>(qmap, kmap, vmap, omap, p, smem, sh, ItemSource{nullptr, nullptr, 0u});
}

// Plan area of the workspace (after the decode part):
//   [0] n_tiles int32, [8] plan flag u64, [16] item counter u64 (padded to 256 bytes),
//   [256] cost histogram int32 [PLAN_MAX_COST + 1] (padded to 256), then the tile list int2 [...].
// Costs (key tiles of a query tile) above PLAN_MAX_COST share its bucket: only the order
// among such tiles is affected.
constexpr int PLAN_MAX_COST = 12000;
constexpr size_t PLAN_HIST_BYTES = ((size_t)(PLAN_MAX_COST + 1) * 4 + 255) / 256 * 256;

struct PlanArea {
    int32_t* n_tiles;
    unsigned long long* flag;
    unsigned long long* counter;
    int32_t* hist;
    int2* tiles;
};

inline PlanArea plan_area(void* base) {
    uint8_t* b = static_cast<uint8_t*>(base);
    return PlanArea{reinterpret_cast<int32_t*>(b), reinterpret_cast<unsigned long long*>(b + 8),
                    reinterpret_cast<unsigned long long*>(b + 16), reinterpret_cast<int32_t*>(b + 256),
                    reinterpret_cast<int2*>(b + 256 + PLAN_HIST_BYTES)};
}

inline size_t plan_bytes(int batch, int total_q) {
    const size_t nt_max = (size_t)(total_q + BM - 1) / BM + (size_t)batch;
    return 256 + PLAN_HIST_BYTES + nt_max * sizeof(int2);
}

// Host launcher of the one-launch mixed step (mixed.cu): the split-K decode of the entries
// with q_len <= kDecodeMaxQ and the prefill of the others in one persistent kernel, then
// the merge of the split decode segments.  `prm` is the prefill's parameter block (tile
// list in `plan`), the maps as for prefill_kernel.
int launch_fused(int head_dim, cudaStream_t st, void* out, float* lse, const void* q, const void* k_pool,
                 const void* v_pool, int num_pages, const int32_t* block_table, int max_pages_per_seq,
                 const int32_t* cu_seqlens_q, const int32_t* seq_lens, int batch, int total_q, int max_seq_len,
                 int page_size, int num_q_heads, int num_kv_heads, float softmax_scale, void* workspace,
                 size_t dec_bytes, int32_t* status, const CUtensorMap& qmap, const CUtensorMap& kmap,
                 const CUtensorMap& vmap, const CUtensorMap& omap, const Params& prm, const PlanArea& plan,
                 int max_cost);

}  // namespace pf
}  // namespace pa
