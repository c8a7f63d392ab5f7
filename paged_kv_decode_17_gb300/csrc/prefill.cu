// Varlen causal prefill over a paged KV cache on tcgen05 tensor cores.
//
// What it computes ("The Stack Below the Stack, Part 2", section 2.1; "8.
// Kernels and Attention Backends", section "Attention is an I/O problem"):
// exact softmax attention, tiled.  Query tiles of 128 rows and key tiles of 64
// keys stream through on-chip memory; each row carries a running maximum and
// a running sum of exponentials, and the output accumulated so far is
// rescaled when the maximum grows, so the result equals the untiled softmax.
// Row i of a sequence with q_len rows and seq_len keys sits at position
// seq_len - q_len + i and sees keys 0 .. that position.
//
// GB300 design (one CTA = one 128-row query tile of one sequence, for two
// query heads that share a KV head, so each K/V tile is loaded once for both):
// * warp 16 (producer): loads the two Q tiles once by TMA, then gathers K and
//   V tiles through an 8-stage ring: a 64-key tile is four 16-row page blocks
//   found through the block table (one tile ahead), copied with coalesced
//   16-byte cp.async into the 128-byte-swizzled operand layout.
// * warps 17 / 18 (MMA, one per head): one thread issues tcgen05.mma:
//   S_h = Q_h K^T into TMEM (fp32, 64 columns) and O_h += P_h V into TMEM
//   (fp32, D columns).  The issue order S(j+1), PV(j) lets the tensor core
//   compute the next scores while the softmax of the current tile runs.
// * warps 0-15 (softmax): per head two warpgroups, each owning half of the
//   64 score columns of every row (thread = TMEM lane = row); the two halves
//   exchange their row maxima through shared memory at a named barrier.  They
//   write P (bf16 pairs) into TMEM with tcgen05.st, where the P.V MMA reads it
//   as its A operand (no shared-memory round trip, no proxy fence), and at the
//   end normalise O and store it.  O is rescaled only when a row's maximum grows by
//   more than TAU = 8 (log2 units): until then the exponentials are taken
//   against the older, smaller maximum, which keeps them <= 2^8 and the result
//   exact, because the final division uses the same reference maximum for
//   numerator and denominator.
// Every wait is bounded; a timeout sets a CTA-wide abort flag, records
// PA_ERR_TIMEOUT and all roles fall through to a clean exit.
#include "pa_common.cuh"
#include "pa_host.h"

namespace pa {
namespace pf {

constexpr int BM = 128;      // query rows per tile (= TMEM lanes)
constexpr int BN = 64;       // keys per KV tile
#ifndef PA_PF_NSTAGE
#define PA_PF_NSTAGE 8
#endif
#ifndef PA_PF_NPB
#define PA_PF_NPB 2
#endif
#ifndef PA_PF_MAX_CLUSTER
#define PA_PF_MAX_CLUSTER 4
#endif
constexpr int NSTAGE = PA_PF_NSTAGE;  // K/V ring depth (K and V tiles alternate)
constexpr int NPB = PA_PF_NPB;        // P buffers per head (tile j uses buffer j % NPB)
// CTAs of one (sequence, query tile, KV head) -- its head pairs -- form a cluster
// of up to this many; each K/V tile is fetched once per cluster (TMA multicast)
constexpr int MAX_CLUSTER = PA_PF_MAX_CLUSTER;
constexpr float TAU = 8.f;   // rescale threshold, log2 units
// warps 0-15: softmax (head = warp / 8, column half = (warp / 4) & 1, row quarter = warp & 3)
// warp 16: TMA producer; warps 17 and 18: MMA issuers of head 0 and head 1
constexpr int NTHREADS = 608;
constexpr int WARP_TMA = 16, WARP_MMA0 = 17;
constexpr int HALF = BN / 2;  // score columns per softmax thread

template <int D>
struct Cfg {
    static constexpr int KB = D / 64;               // 128-byte column blocks per row
    static constexpr int Q_BYTES = BM * D * 2;      // one head's Q tile
    static constexpr int KV_BYTES = BN * D * 2;     // one K or V tile
    static constexpr int P_BYTES = BM * BN * 2;     // one P tile
    static constexpr int Q_KB = BM * 128;           // bytes per column block of a Q tile
    static constexpr int KV_KB = BN * 128;          // bytes per column block of a K/V tile
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = 2 * Q_BYTES;
    static constexpr int SMEM_BYTES = 1024 + OFF_KV + NSTAGE * KV_BYTES;
    // TMEM columns: S[head] (BN fp32), O[head] (D fp32), P[head][buffer] (BN bf16 = BN/2)
    static constexpr int TM_S0 = 0;
    static constexpr int TM_O0 = 2 * BN;
    static constexpr int TM_P0 = 2 * BN + 2 * D;
    static constexpr int TM_USED = TM_P0 + 2 * NPB * (BN / 2);
    static constexpr int TM_COLS = TM_USED <= 256 ? 256 : 512;
    static_assert(TM_USED <= 512, "TMEM budget");
    static constexpr uint32_t IDESC_S = tc::idesc_bf16(BM, BN, 0, 0);   // Q K-major, K K-major
    static constexpr uint32_t IDESC_PV = tc::idesc_bf16(BM, D, 0, 1);   // P K-major, V MN-major
};

struct Params {
    __nv_bfloat16* out;
    float* lse;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* cu_q;
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    int32_t* status;
    int num_pages, max_pages, batch, page_size;
    int Hq, Hkv, group, NP;  // NP = head pairs per KV head, padded to a multiple of CS
    int CS;                  // cluster size (CTAs sharing each K/V tile)
    int skip_single;  // sequences with q_len == 1 are served by the decode kernel
    float scale_log2;
};

struct Shared {
    uint64_t bar_q;
    uint64_t kv_full[NSTAGE];
    uint64_t kv_empty[NSTAGE];
    uint64_t s_full[2], s_free[2];
    uint64_t p_ready[2][NPB], pv_done[2][NPB];  // [head][P buffer]
    uint64_t v_tail;  // TMA copies of a V tile that runs past the sequence end land here first
    float xmax[2][2][2][BM];  // [head][tile parity][column half][row]: partial row maxima
    float xsum[2][2][BM];     // [head][column half][row]: partial row sums at the end
    uint32_t tmem_base;
    int abort_flag;
    int item[9];
};

__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, Shared& sh, int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(&sh.abort_flag)) return false;
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
            report(status, PA_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_mc(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                               uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "h"(mask)
        : "memory");
}

// Arrive on `bar` at the same offset in every CTA of `mask` once this thread's MMAs are done.
__device__ __forceinline__ void commit_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// number of 128-row tiles of sequence b served by this kernel (0 if none)
__device__ __forceinline__ int seq_tiles(const Params& p, int b, int& q_len, int& seq_len) {
    q_len = __ldg(p.cu_q + b + 1) - __ldg(p.cu_q + b);
    seq_len = __ldg(p.seq_lens + b);
    if (q_len < 0 || seq_len < q_len || seq_len > p.max_pages * p.page_size) {
        report(p.status, PA_ERR_BAD_LEN);
        return 0;
    }
    if (q_len == 0 || (p.skip_single && q_len == 1)) return 0;
    return (q_len + BM - 1) / BM;
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const Params p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Shared sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // ---- which (sequence, tile, KV head, head pair) this CTA computes
    if (warp == 0) {
        const int per = p.Hkv * p.NP;
        const int T = blockIdx.x / per;
        const int rem = blockIdx.x - T * per;
        int found_b = -1, found_P = 0, found_n = 0, P = 0;
        for (int b0 = 0; b0 < p.batch && found_b < 0; b0 += 32) {
            const int b = b0 + lane;
            int ql = 0, sl = 0, n = 0;
            if (b < p.batch) n = seq_tiles(p, b, ql, sl);
            const int incl = warp_incl_scan(n);
            const int tot = __shfl_sync(0xffffffffu, incl, 31);
            if (T < P + tot) {
                const unsigned hit = __ballot_sync(0xffffffffu, P + incl > T);
                const int l = __ffs(hit) - 1;
                found_b = b0 + l;
                found_P = P + __shfl_sync(0xffffffffu, incl - n, l);
                found_n = __shfl_sync(0xffffffffu, n, l);
            }
            P += tot;
        }
        if (lane == 0) {
            sh.item[0] = found_b;
            if (found_b >= 0) {
                const int g = rem / p.NP;
                const int pair = rem - g * p.NP;
                const int ql = __ldg(p.cu_q + found_b + 1) - __ldg(p.cu_q + found_b);
                const int sl = __ldg(p.seq_lens + found_b);
                const int t = found_n - 1 - (T - found_P);  // heaviest tile of the sequence first
                sh.item[1] = t;
                sh.item[2] = ql;
                sh.item[3] = sl;
                sh.item[4] = __ldg(p.cu_q + found_b) + t * BM;    // first q row of the tile
                sh.item[5] = g;
                sh.item[6] = g * p.group + 2 * pair;                       // first query head
                sh.item[7] = max(0, min(2, p.group - 2 * pair));           // heads in this CTA (0: loads only)
                const int pair0 = pair - pair % p.CS;                       // first pair of the cluster
                sh.item[8] = max(0, min(2 * p.CS, p.group - 2 * pair0));   // heads in the cluster
            }
            sh.abort_flag = 0;
        }
    }
    __syncthreads();
    if (tid == 0) {
        mbar_init(&sh.bar_q, 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&sh.kv_full[s], 1);
            // released once by every head of the cluster (each MMA thread commits to all CTAs)
            mbar_init(&sh.kv_empty[s], sh.item[0] >= 0 ? max(1, sh.item[8]) : 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&sh.s_full[h], 1);
            mbar_init(&sh.s_free[h], 8 * 32);
            mbar_init(&sh.v_tail, 1);
            for (int bf = 0; bf < NPB; ++bf) {
                mbar_init(&sh.p_ready[h][bf], 8 * 32);
                mbar_init(&sh.pv_done[h][bf], 1);
            }
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (sh.item[0] < 0) return;  // uniform over the cluster: no tile for it
    const int CS = p.CS;
    const uint16_t cmask = (uint16_t)((1u << CS) - 1);
    const int crank = CS > 1 ? (int)cluster_rank() : 0;
    if (CS > 1) cluster_sync();  // every CTA's barriers exist before anyone multicasts into them

    const int b = sh.item[0];
    const int t = sh.item[1];
    const int q_len = sh.item[2];
    const int seq_len = sh.item[3];
    const int row0 = sh.item[4];
    const int g = sh.item[5];
    const int h0 = sh.item[6];
    const int nheads = sh.item[7];
    const int prior = seq_len - q_len;
    const int rows_valid = min(BM, q_len - t * BM);
    const int qmin = prior + t * BM;                 // position of the tile's first row
    const int qlast = qmin + rows_valid - 1;         // position of its last valid row
    const int n_kv = qlast / BN + 1;                 // key tiles 0 .. n_kv-1

    if (warp == WARP_TMA) {
        tc::tmem_alloc(&sh.tmem_base, C::TM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh.tmem_base;

    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sKV = smem + C::OFF_KV;

    if (warp == WARP_TMA) {
        // ===================================================== producer (whole warp)
        if (lane == 0) {
            prefetch_tensormap(&qmap);
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            if (nheads > 0) {
                mbar_arrive_expect_tx(&sh.bar_q, nheads * C::Q_BYTES);
                for (int hh = 0; hh < nheads; ++hh)
                    for (int kb = 0; kb < C::KB; ++kb)
                        tma_load_3d(sQ + hh * C::Q_BYTES + kb * C::Q_KB, &qmap, &sh.bar_q, kb * 64, h0 + hh, row0);
            }
        }
        // A K (or V) tile is 4 x KB boxes: 16-key page blocks x 64-column halves.  Box b
        // is fetched by the cluster CTA of rank b % CS and multicast to all of them, so
        // every CTA's barrier receives the whole tile.  Lane u < 4 resolves block u of a
        // tile through the block table one tile ahead.
        const int32_t* bt = p.block_table + (size_t)b * p.max_pages;
        auto block_row = [&](int j) -> int {  // pool row of block `lane` of tile j, -1 if none
            int row = -1;
            if (lane < 4 && j < n_kv) {
                const int key0 = j * BN + lane * 16;
                if (key0 < seq_len) {
                    const int page = key0 / p.page_size;
                    const int phys = __ldg(bt + page);
                    if (phys < 0 || phys >= p.num_pages)
                        report(p.status, PA_ERR_BAD_PAGE);
                    else
                        row = (phys * p.Hkv + g) * p.page_size + (key0 - page * p.page_size);
                }
            }
            return row;
        };
        int next_row = block_row(0);
        bool ok = true;
        int issued = 0;
        for (int j = 0; j < n_kv && ok; ++j) {
            const int my_row = next_row;
            next_row = block_row(j + 1);
            const unsigned goodmask = __ballot_sync(0xffffffffu, my_row >= 0) & 0xFu;
            const int good = __popc(goodmask);
            const int box_row = __shfl_sync(0xffffffffu, my_row, (lane / C::KB) & 3);  // block of box `lane`
            const bool mine = lane < 4 * C::KB && (lane % CS) == crank && box_row >= 0;
            const bool tail = (j + 1) * BN > seq_len;
            for (int x = 0; x < 2 && ok; ++x) {
                const int i = 2 * j + x;
                const int st = i % NSTAGE;
                ok = __all_sync(0xffffffffu, wait_ab(&sh.kv_empty[st], ((i / NSTAGE) & 1) ^ 1, sh, p.status));
                if (!ok) break;
                uint8_t* dst = sKV + st * C::KV_BYTES;
                const bool via_tail = (x == 1) && tail;
                uint64_t* land = via_tail ? &sh.v_tail : &sh.kv_full[st];
                if (lane == 0) {
                    if (good == 0)
                        mbar_arrive(land);
                    else
                        mbar_arrive_expect_tx(land, good * 16 * D * 2);  // the whole tile, from all CTAs
                }
                __syncwarp();
                if (mine) {
                    const int u = lane / C::KB, kb = lane - u * C::KB;
                    uint8_t* bdst = dst + kb * C::KV_KB + u * 2048;
                    const CUtensorMap* map = x == 0 ? &kmap : &vmap;
                    if (CS > 1)
                        tma_load_2d_mc(bdst, map, land, kb * 64, box_row, cmask);
                    else
                        tma_load_2d(bdst, map, land, kb * 64, box_row);
                }
                ++issued;
                if (via_tail) {
                    // keys past the sequence end: their V rows may hold anything and 0 * NaN = NaN,
                    // so zero them (in this CTA's copy) before any MMA may read this tile
                    ok = __all_sync(0xffffffffu, wait_ab(&sh.v_tail, 0, sh, p.status));
                    if (!ok) break;
                    const int first = seq_len - j * BN;
                    const int nchunk = (BN - first) * 8 * C::KB;  // 16-byte chunks to clear
                    for (int c = lane; c < nchunk; c += 32) {
                        const int kb = c / ((BN - first) * 8);
                        const int rem = c - kb * (BN - first) * 8;
                        const int r = first + rem / 8;
                        *reinterpret_cast<uint4*>(dst + kb * C::KV_KB + r * 128 + (rem & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.kv_full[st]);
                }
            }
        }
        // Before leaving: every copy into this CTA has landed and every head of the
        // cluster has released the last stages (no remote arrival can still target us).
        if (lane == 0) {
            if (nheads > 0) mbar_wait(&sh.bar_q, 0);
            for (int i = max(0, issued - NSTAGE); i < issued; ++i) {
                mbar_wait(&sh.kv_full[i % NSTAGE], (i / NSTAGE) & 1);
                mbar_wait(&sh.kv_empty[i % NSTAGE], (i / NSTAGE) & 1);
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA0 || warp == WARP_MMA0 + 1) {
        // ===================================================== MMA issuer of one head
        const int hh = warp - WARP_MMA0;
        if (lane == 0 && hh < nheads) {
            const uint32_t qaddr = smem_u32(sQ) + hh * C::Q_BYTES;
            const uint32_t t_p = tmem + C::TM_P0 + hh * NPB * (BN / 2);
            const uint32_t kv_base = smem_u32(sKV);
            const uint32_t t_s = tmem + C::TM_S0 + hh * BN;
            const uint32_t t_o = tmem + C::TM_O0 + hh * D;
            bool ok = wait_ab(&sh.bar_q, 0, sh, p.status);
            tc::fence_after_sync();
            auto issue_s = [&](int j) {
                const uint32_t kaddr = kv_base + ((2 * j) % NSTAGE) * C::KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad = tc::smem_desc_sw128(qaddr + (kk >> 2) * C::Q_KB + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(kaddr + (kk >> 2) * C::KV_KB + (kk & 3) * 32, 16, 1024);
                    tc::mma_ss(t_s, ad, bd, C::IDESC_S, kk > 0);
                }
                tc::commit(&sh.s_full[hh]);
            };
            auto issue_pv = [&](int j) {
                const uint32_t vaddr = kv_base + ((2 * j + 1) % NSTAGE) * C::KV_BYTES;
                const uint32_t pcol = t_p + (j % NPB) * (BN / 2);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bd = tc::smem_desc_sw128(vaddr + kk * 2048, C::KV_KB, 1024);
                    tc::mma_ts(t_o, pcol + kk * 8, bd, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(&sh.pv_done[hh][j % NPB]);
            };
            // a K/V stage is free once every head of the cluster is done with it
            auto release = [&](uint64_t* bar) {
                if (CS > 1)
                    commit_mc(bar, cmask);
                else
                    tc::commit(bar);
            };
            // prologue: scores of key tile 0
            if (ok) ok = wait_ab(&sh.kv_full[0], 0, sh, p.status);
            if (ok) {
                tc::fence_after_sync();
                issue_s(0);
                release(&sh.kv_empty[0]);
            }
            for (int j = 0; j < n_kv && ok; ++j) {
                const int ik = 2 * (j + 1), iv = 2 * j + 1;
                if (j + 1 < n_kv) {
                    // next scores as soon as the softmax has pulled the current ones out of TMEM
                    ok = wait_ab(&sh.kv_full[ik % NSTAGE], (ik / NSTAGE) & 1, sh, p.status) &&
                         wait_ab(&sh.s_free[hh], j & 1, sh, p.status);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_s(j + 1);
                    release(&sh.kv_empty[ik % NSTAGE]);
                }
                ok = wait_ab(&sh.kv_full[iv % NSTAGE], (iv / NSTAGE) & 1, sh, p.status) &&
                     wait_ab(&sh.p_ready[hh][j % NPB], (j / NPB) & 1, sh, p.status);
                if (!ok) break;
                tc::fence_after_sync();
                issue_pv(j);
                release(&sh.kv_empty[iv % NSTAGE]);
            }
        }
        __syncwarp();
    } else {
        // ===================================================== softmax (thread = row, half the columns)
        const int hh = warp >> 3;
        const int half = (warp >> 2) & 1;
        if (hh < nheads) {
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;  // tile row = TMEM lane
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const uint32_t t_s = tmem + lane_off + C::TM_S0 + hh * BN + half * HALF;
            const uint32_t t_o = tmem + lane_off + C::TM_O0 + hh * D + half * (D / 2);
            const uint32_t t_p = tmem + lane_off + C::TM_P0 + hh * NPB * (BN / 2);
            const int qpos = qmin + r;
            const int key_off = half * HALF;
            float m_ref = -INFINITY, l = 0.f;
            // `ok` turns false (for the whole warp) once a wait times out or another role
            // aborted; the loop still runs to the end so that both column halves of a head
            // meet at every named barrier, but does no further work
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                if (ok) ok = __all_sync(0xffffffffu, wait_ab(&sh.s_full[hh], j & 1, sh, p.status));
                float x[HALF];
                float mine = -INFINITY;
                if (ok) {
                    tc::fence_after_sync();
                    uint32_t sr[HALF];
                    tc::ld_32x32b_x32(t_s, sr);
                    tc::wait_ld();
                    tc::fence_before_sync();
                    mbar_arrive(&sh.s_free[hh]);
#pragma unroll
                    for (int c = 0; c < HALF; ++c) x[c] = __uint_as_float(sr[c]);
                    if ((j + 1) * BN - 1 > qmin) {  // diagonal tile: some key is after some row
                        const int k0 = j * BN + key_off;
#pragma unroll
                        for (int c = 0; c < HALF; ++c)
                            if (k0 + c > qpos) x[c] = -INFINITY;
                    }
                    // row max of the raw scores (softmax_scale > 0) over my half, as a tree
                    float t8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) t8[i] = x[i];
#pragma unroll
                    for (int c = 8; c < HALF; ++c) t8[c & 7] = fmaxf(t8[c & 7], x[c]);
                    mine = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                                 fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
                }
                // exchange with the warp holding the other half of the row
                sh.xmax[hh][j & 1][half][r] = mine;
                asm volatile("bar.sync %0, %1;" ::"r"(1 + hh), "r"(8 * 32) : "memory");
                if (ok) ok = !*reinterpret_cast<volatile int*>(&sh.abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) continue;
                const float other = sh.xmax[hh][j & 1][half ^ 1][r];
                const float mx = (half == 0 ? fmaxf(mine, other) : fmaxf(other, mine)) * p.scale_log2;
                if (j == 0) {
                    m_ref = mx;
                } else if (__any_sync(0xffffffffu, mx > m_ref + TAU)) {
                    // rescale O (this half's columns) to a new reference maximum
                    const float m_new = fmaxf(m_ref, mx);
                    const float alpha = ex2(m_ref - m_new);
                    // all earlier PVs are done once PV(j-1) is (one issuing thread, in order)
                    ok = __all_sync(0xffffffffu,
                                    wait_ab(&sh.pv_done[hh][(j - 1) % NPB], ((j - 1) / NPB) & 1, sh, p.status));
                    if (!ok) continue;
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c0 = 0; c0 < D / 2; c0 += 32) {
                        uint32_t o[32];
                        tc::ld_32x32b_x32(t_o + c0, o);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc::st_32x32b_x32(t_o + c0, o);
                    }
                    tc::wait_st();
                    l *= alpha;
                    m_ref = m_new;
                }
                // p = 2^(s * scale_log2 - m_ref): one FFMA + one MUFU each; partial sums as a tree
                const float neg = -m_ref;
                float s8[8];
                uint32_t pk[HALF / 2];
#pragma unroll
                for (int c = 0; c < HALF; c += 2) {
                    const float p0 = ex2(fmaf(x[c], p.scale_log2, neg));
                    const float p1 = ex2(fmaf(x[c + 1], p.scale_log2, neg));
                    const int k = (c >> 1) & 7;
                    s8[k] = (c < 16) ? (p0 + p1) : (s8[k] + (p0 + p1));
                    pk[c >> 1] = pack_bf16x2(p0, p1);
                }
                l += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
                // P buffer j % NPB was last read by PV(j - NPB).  Waiting for that also keeps
                // each p_ready / pv_done barrier within one phase of its waiter (mbarrier
                // parity only tells adjacent phases apart).
                if (j >= NPB) {
                    ok = __all_sync(0xffffffffu,
                                    wait_ab(&sh.pv_done[hh][j % NPB], ((j / NPB) - 1) & 1, sh, p.status));
                    if (!ok) continue;
                }
                // P (bf16 pairs, low half = even key) into this head's TMEM P columns
                tc::st_32x32b_x16(t_p + (j % NPB) * (BN / 2) + half * (HALF / 2), pk);
                tc::wait_st();
                tc::fence_before_sync();
                mbar_arrive(&sh.p_ready[hh][j % NPB]);
            }
            // ---- epilogue: O / l -> bf16, each half stores its D/2 columns
            sh.xsum[hh][half][r] = l;
            asm volatile("bar.sync %0, %1;" ::"r"(1 + hh), "r"(8 * 32) : "memory");
            const float lt = half == 0 ? l + sh.xsum[hh][1][r] : sh.xsum[hh][0][r] + l;
            if (ok)
                ok = __all_sync(0xffffffffu,
                                wait_ab(&sh.pv_done[hh][(n_kv - 1) % NPB], ((n_kv - 1) / NPB) & 1, sh, p.status));
            if (ok) {
                tc::fence_after_sync();
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                const bool store = r < rows_valid;
                const int h = h0 + hh;
                __nv_bfloat16* orow = p.out + ((size_t)(row0 + r) * p.Hq + h) * D + half * (D / 2);
#pragma unroll 1
                for (int c0 = 0; c0 < D / 2; c0 += 32) {
                    uint32_t o[32];
                    tc::ld_32x32b_x32(t_o + c0, o);
                    tc::wait_ld();
                    if (store) {
                        uint32_t pkd[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pkd[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
                    }
                }
                if (store && half == 0 && p.lse != nullptr)
                    p.lse[(size_t)(row0 + r) * p.Hq + h] = lt > 0.f ? (m_ref + lg2(lt)) * kLn2 : -INFINITY;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (CS > 1) cluster_sync();  // nobody multicasts into or arrives on this CTA any more
    tc::fence_after_sync();
    if (warp == WARP_TMA) tc::tmem_dealloc(tmem, C::TM_COLS);
}

}  // namespace pf
}  // namespace pa

using namespace pa;

extern "C" size_t pa_prefill_workspace_bytes(int batch, int total_q, int num_q_heads, int num_kv_heads,
                                             int head_dim) {
    (void)total_q;
    return pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim);
}

extern "C" int attn_prefill_varlen_causal(void* out, float* lse, const void* q, const void* k_pool,
                                          const void* v_pool, int num_pages, const int32_t* block_table,
                                          int max_pages_per_seq, const int32_t* cu_seqlens_q,
                                          const int32_t* seq_lens, int batch, int total_q, int max_q_len,
                                          int max_seq_len, int page_size, int num_q_heads, int num_kv_heads,
                                          int head_dim, float softmax_scale, void* workspace,
                                          size_t workspace_bytes, int32_t* status, void* stream) {
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

    const int group = num_q_heads / num_kv_heads;
    const int pairs = (group + 1) / 2;
    const int CS = pairs < pf::MAX_CLUSTER ? pairs : pf::MAX_CLUSTER;
    const int NP = (pairs + CS - 1) / CS * CS;  // padded: a cluster never spans two KV heads
    const long long tiles_upper = (long long)(total_q + pf::BM - 1) / pf::BM + batch;
    const long long grid = tiles_upper * num_kv_heads * NP;
    if (grid >= (1ll << 31)) return PA_ERR_SHAPE;

    CUtensorMap qmap, kmap, vmap;
    if (encode_q_map(&qmap, q, total_q, num_q_heads, head_dim) != PA_OK) return PA_ERR_CUDA;
    if (encode_rows_map(&kmap, k_pool, (uint64_t)pool_rows, head_dim, 64, 16) != PA_OK) return PA_ERR_CUDA;
    if (encode_rows_map(&vmap, v_pool, (uint64_t)pool_rows, head_dim, 64, 16) != PA_OK) return PA_ERR_CUDA;

    pf::Params prm;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.block_table = block_table;
    prm.seq_lens = seq_lens;
    prm.cu_q = cu_seqlens_q;
    prm.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
    prm.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
    prm.status = status;
    prm.num_pages = num_pages;
    prm.max_pages = max_pages_per_seq;
    prm.batch = batch;
    prm.page_size = page_size;
    prm.Hq = num_q_heads;
    prm.Hkv = num_kv_heads;
    prm.group = group;
    prm.NP = NP;
    prm.CS = CS;
    prm.skip_single = 1;  // q_len == 1 entries go to the split-K decode kernel below
    prm.scale_log2 = softmax_scale * kLog2e;

    // decode rows (q_len == 1) of a mixed step: split-K over their KV
    rc = dec::launch_decode(out, lse, q, k_pool, v_pool, num_pages, block_table, max_pages_per_seq, seq_lens,
                            cu_seqlens_q, batch, max_seq_len, page_size, num_q_heads, num_kv_heads, head_dim,
                            softmax_scale, workspace, workspace_bytes, status, stream);
    if (rc != PA_OK) return rc;
    if (max_q_len < 2) return PA_OK;  // no entry needs the prefill kernel

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(pf::NTHREADS, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    if (head_dim == 128) {
        cfg.dynamicSmemBytes = pf::Cfg<128>::SMEM_BYTES;
        if (set_smem_limit_once((const void*)pf::prefill_kernel<128>, pf::Cfg<128>::SMEM_BYTES, dev.device, 2) !=
            PA_OK)
            return PA_ERR_CUDA;
        err = cudaLaunchKernelEx(&cfg, pf::prefill_kernel<128>, qmap, kmap, vmap, prm);
    } else {
        cfg.dynamicSmemBytes = pf::Cfg<64>::SMEM_BYTES;
        if (set_smem_limit_once((const void*)pf::prefill_kernel<64>, pf::Cfg<64>::SMEM_BYTES, dev.device, 3) !=
            PA_OK)
            return PA_ERR_CUDA;
        err = cudaLaunchKernelEx(&cfg, pf::prefill_kernel<64>, qmap, kmap, vmap, prm);
    }
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
