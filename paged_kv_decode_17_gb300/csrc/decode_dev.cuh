// Split-K paged decode: Flash-Decoding over a paged KV cache (device code).
//
// What it computes ("The Stack Below the Stack, Part 2", section 2.2
// Flash-Decoding): the KV sequence of every (sequence, KV head) is split into
// chunks; each chunk yields a normalised partial output and its local
// log-sum-exp; the chunks are merged with
//     lse = log sum_c exp(lse_c),   o = sum_c exp(lse_c - lse) o_c.
// Inside a chunk, keys are streamed 16 at a time with the online softmax of
// section 2.1 (running max and running sum, rescaled when the max grows).
//
// GB300 design
// * Work is measured in "units": 16 consecutive tokens of one row block of a
//   (sequence b, KV head g, row segment sb) segment (row blocks below).  A
//   unit is one 16 x D bf16 block of K plus one of V, contiguous in the
//   [page][Hkv][page_size][D] pools.  All units of all segments are laid end to end and every CTA of a
//   persistent grid (a multiple of the SM count) takes one equal contiguous
//   range of them, so a 1-token sequence and a 131k-token one balance the
//   same way.  The ranges are derived on the device from seq_lens (no host
//   synchronisation; the call can be captured in a CUDA graph).
// * Inside a CTA each warp takes every W-th unit of the CTA's part of a
//   segment and runs its own copy pipeline: DEPTH stages, each unit's K and V
//   staged by 16-byte cp.async copies (coalesced 512-byte warp requests) into a
//   128-byte-swizzled layout, so the ldmatrix reads below are bank-conflict
//   free.  (Per-thread copies, not TMA: with one 16-row page block per request,
//   the TMA engine's per-request cost capped the read rate near 18 bytes per
//   cycle per SM.)  There is no cross-warp producer/consumer handshake in the
//   loop.
// * Q.K^T and P.V run on bf16 mma.sync (m16n8k16) with query rows as the M
//   dimension: the rows of one (sequence, KV head) are its q_len query tokens
//   times the GQA group's heads (numbered token-major), cut into row blocks of
//   at most 16.  Up to 4 row blocks (64 rows) form one segment; its units are
//   ordered key block by key block, row block fastest, so the warps that take
//   the row blocks of one key block stage it at the same moment and all but
//   the first find it in L2.  With q_len > 1 (multi-query decode, e.g. the
//   verification of speculated tokens) row i of the query block sees keys
//   0 .. seq_len - q_len + i.  Scores, running max/sum and O stay in fp32
//   registers; O is rescaled only when a row's maximum grows by more than
//   kDecTau (conditional rescaling, "The Stack Below the Stack, Part 2",
//   section 2.3).
// * At the end of the CTA's part of a segment the states of the warps that
//   hold the same row block are merged in shared memory in a fixed order.  A
//   segment covered by one chunk is normalised and stored directly; otherwise
//   the partial (o_c, lse_c) goes to the workspace slot of its chunk, and a
//   second, small kernel (launched as a programmatic dependent of the first)
//   merges each split segment's partials in chunk order, one thread per
//   (row, 4 dimensions), so results are bit-identical run to run.  (Merging
//   in the decode kernel, by the last CTA to finish a segment, held that CTA
//   up for several L2 round trips at the very end of its range: the CTAs that
//   merged set the length of the whole launch.)
#pragma once

#include "pa_common.cuh"
#include "pa_host.h"

#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace pa {
namespace dec {

constexpr int W = 4;           // warps per CTA
constexpr int UNIT = 16;       // tokens per unit
constexpr int RB = 16;         // rows per row block (mma M)
constexpr int SBR = 64;        // rows per segment (at most W row blocks)
constexpr int MIN_CHUNK = 16;  // minimum units per CTA
// Conditional rescaling (log2 units): a row's reference maximum moves only when a
// unit's scores exceed it by more than this, so the exponentials stay <= 2^8 and O and
// l are rescaled rarely.  The result is unchanged: numerator and denominator are taken
// against the same reference.
constexpr float kDecTau = 8.f;
// CTAs (of 4 warps) per SM: they hide each other's latency.  The swapped-operand
// FP8 variant is bound by its own instruction latency and runs three per SM (in
// 168 registers, with shallower staging so the shared memory fits); the others
// run two (the bf16 decode loses more to the register cap than it gains).
template <bool FP8, bool SWAP>
constexpr int ctas_per_sm() { return (FP8 && SWAP) ? 3 : 2; }
constexpr int kMaxCtasPerSM = 3;  // sizes the workspace slots for either grid

// Per-warp copy pipeline depth (units in flight); the three-per-SM variant gets
// the shallower pipeline.
template <int D, bool FP8 = false, bool SWAP = false>
struct Cfg {
    static constexpr int DEPTH = FP8 ? (SWAP ? 3 : 6) : (D == 128 ? 3 : 6);
    static constexpr int BOXES = D / 64;             // 128-byte-wide column blocks per row (bf16)
    static constexpr int BOX_BYTES = UNIT * 128;     // 16 rows x 128 bytes
    static constexpr int UNIT_BYTES = UNIT * D * (FP8 ? 1 : 2);  // one K or V unit
    static constexpr int STAGE_BYTES = 2 * UNIT_BYTES;
    static constexpr int STAGES_BYTES = W * DEPTH * STAGE_BYTES;
    static constexpr int MSTRIDE = D + 4;  // fp32 row stride of the merge buffer
    static constexpr int MERGE_BYTES = RB * MSTRIDE * 4;  // warps add into it one after another
    static constexpr int SMEM_BYTES = 1024 + STAGES_BYTES + MERGE_BYTES;
};

struct Params {
    __nv_bfloat16* out;
    float* lse;
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_pool;  // FP8 variant: e4m3 codes, [page][Hkv][page_size][D]
    const __nv_bfloat16* v_pool;  // FP8 variant: e4m3 codes, [page][Hkv][D][page_size] (transposed)
    const __nv_bfloat16* k_new;   // append (bf16 only): K/V rows of the query tokens, [rows][Hkv][D],
    const __nv_bfloat16* v_new;   // read in place of their pool slots and written there; null: none
    __nv_bfloat16* k_pool_w;      // append: the pools, writable
    __nv_bfloat16* v_pool_w;
    const float* k_scale;         // FP8 variant: [Hkv], K = code * k_scale[g]
    const float* v_scale;         // FP8 variant: [Hkv], V = code * v_scale[g]
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* cu_q;  // null: one query row per sequence (row b); else rows cu_q[b] .. cu_q[b+1]
    int32_t* seg_base;  // [batch + 1]: first unit of each sequence, then the total (written by CTA 0)
    int G;              // CTAs of the decode grid
    float* ws_lse;  // [slots][RS], log2 domain
    float* ws_o;    // [slots][RS][D], normalised
    int32_t* status;
    int num_pages, max_pages, batch, page_size, ps_shift;  // page_size = 1 << ps_shift
    int total_q;  // rows of q / out
    int qmax;     // entries with 1 <= q_len <= qmax are served here
    int qcap;     // q_len in (qmax, qcap] is an error (larger ones belong to the prefill kernel)
    int Hq, Hkv, group;
    int SBmax;    // segments per (sequence, KV head) at q_len = qmax
    int RS;       // rows per workspace slot (16 x the largest row-block count)
    int min_chunk;  // smallest chunk, in units (MIN_CHUNK unless overridden for tests)
    unsigned long long* reset_words;  // null, or 2 words the merge kernel zeroes once the decode grid is done
    float scale_log2;
};

// Row geometry of one served sequence: rows = q_len * group, split into SB
// segments of RSB rows, each split into 1 << nrb_shift row blocks of R rows.
struct SeqShape {
    int len, qlen, nkb, SB, RSB, nrb_shift, R;
};

__device__ __forceinline__ SeqShape seq_shape(const Params& p, int b) {
    SeqShape s;
    s.len = 0;
    s.nkb = 0;
    s.SB = 1;
    s.RSB = 0;
    s.nrb_shift = 0;
    s.R = 0;
    s.qlen = 1;
    if (p.cu_q != nullptr) {
        const int c0 = __ldg(p.cu_q + b), c1 = __ldg(p.cu_q + b + 1);
        s.qlen = c1 - c0;
        if (c0 < 0 || c1 > p.total_q || (s.qlen > p.qmax && s.qlen <= p.qcap)) {
            report(p.status, PA_ERR_BAD_LEN);
            s.qlen = 0;
        }
        if (s.qlen < 1 || s.qlen > p.qmax) {
            s.qlen = 0;  // not served by this kernel
            return s;
        }
    }
    int len = __ldg(p.seq_lens + b);
    const int cap = p.max_pages * p.page_size;
    if (len < 0 || len > cap || (s.qlen > 1 && len < s.qlen)) {
        report(p.status, PA_ERR_BAD_LEN);
        len = len < 0 ? 0 : (len > cap ? cap : len);
    }
    s.len = len;
    s.nkb = (len + UNIT - 1) / UNIT;
    const int rows = s.qlen * p.group;
    s.SB = (rows + SBR - 1) / SBR;
    s.RSB = (rows + s.SB - 1) / s.SB;
    const int nrb = (s.RSB + RB - 1) / RB;
    s.nrb_shift = nrb <= 1 ? 0 : (nrb == 2 ? 1 : 2);
    s.R = (s.RSB + (1 << s.nrb_shift) - 1) >> s.nrb_shift;
    return s;
}

// Units of all segments of sequence b.
__device__ __forceinline__ int seq_units(const Params& p, const SeqShape& s) {
    return (s.nkb << s.nrb_shift) * p.Hkv * s.SB;
}

// Row of q / out holding token 0 of sequence b's query block.
__device__ __forceinline__ size_t q_row(const Params& p, int b) {
    return p.cu_q == nullptr ? (size_t)b : (size_t)__ldg(p.cu_q + b);
}

// One (b, g, sb) segment: its units are [start, end) in the global order
// b-major, then g, then sb; inside, key block major, row block fastest.
struct Seg {
    int b, g, sb, n, start, end;
    SeqShape sh;
};

__device__ __forceinline__ void seg_set_seq(Seg& s, const Params& p, int b) {
    s.b = b;
    if (b < p.batch) {
        s.sh = seq_shape(p, b);
    } else {
        s.sh.nkb = 0;
        s.sh.SB = 1;
        s.sh.nrb_shift = 0;
    }
    s.n = s.sh.nkb << s.sh.nrb_shift;
}

// Advance to the next segment with at least one unit.  The caller makes sure
// one exists (the CTA's range ends before the last unit).
__device__ __forceinline__ void seg_next(Seg& s, const Params& p) {
    do {
        s.start = s.end;
        if (++s.sb == s.sh.SB) {
            s.sb = 0;
            if (++s.g == p.Hkv) {
                s.g = 0;
                seg_set_seq(s, p, s.b + 1);
            }
        }
        s.end = s.start + s.n;
    } while (s.n == 0 && s.b < p.batch);
}

// The sequence of units one warp loads: within each segment piece
// [pa, pe) of the CTA range, units pa + w, pa + w + W, ...
struct UnitIter {
    Seg seg;
    int pe, u, U1;
    bool done;
    int pc_base;  // page cache: unit whose page lane 0 holds (-1: empty)
    int pc_phys;  // this lane's entry: the page of unit pc_base + lane * W (-1 past the piece)
    __device__ __forceinline__ void norm(const Params& p, int w) {
        while (!done && u >= pe) {
            if (pe >= U1) {
                done = true;
                break;
            }
            seg_next(seg, p);
            pe = min(U1, seg.end);
            u = seg.start + w;
            pc_base = -1;
        }
    }
};

// Physical page of unit it.u.  The warp keeps the pages of its next 32 units,
// one per lane, and reloads all 32 at once (one block_table load per lane, in
// parallel) when it runs past them or enters a new segment, so issuing a unit
// does not wait for a block_table round trip.
__device__ __forceinline__ int unit_page(const Params& p, UnitIter& it, int lane) {
    int k = (it.u - it.pc_base) / W;
    if (it.pc_base < 0 || k >= 32) {
        it.pc_base = it.u;
        const int ul = it.u + lane * W;
        int v = -1;
        if (ul < it.pe) {
            const int j = (ul - it.seg.start) >> it.seg.sh.nrb_shift;  // key block
            v = __ldg(p.block_table + (size_t)it.seg.b * p.max_pages + ((j * UNIT) >> p.ps_shift));
        }
        it.pc_phys = v;
        k = 0;
    }
    return __shfl_sync(0xffffffffu, it.pc_phys, k);
}

// Per-lane parts of the bf16 staging copies' addresses, the same for every unit.
// In step j of K and of V, lane l copies 16-byte chunk cc = l mod CH of row
// r = RPI j + l / CH (CH = D / 8 chunks per row, RPI = 32 / CH rows per step); the
// chunk sits at row * 2D + src in the pool and at RPI j * 128 + dst[j mod SWP] in
// the stage (the 128-byte swizzle of row r only depends on j mod SWP).
// FP8: the K rows are D bytes (CH = D / 16 chunks, RPI = 32 / CH rows per step, 128-byte
// swizzle at D = 128); each lane then copies one 16-byte transposed V row per step.
template <int D, bool FP8 = false>
struct CopyLanes {
    static constexpr int CH = FP8 ? D / 16 : D / 8, RPI = 32 / CH;
    static constexpr int SWP = (FP8 && D != 128) ? 1 : 8 / RPI, STEPS = UNIT / RPI;
    static constexpr int ROW = FP8 ? D : 2 * D;  // bytes per K row
    uint32_t src;
    uint32_t dst[SWP];
    __device__ __forceinline__ explicit CopyLanes(int lane) {
        const int rl = lane / CH, cc = lane % CH;
        src = (uint32_t)(rl * ROW + cc * 16);
#pragma unroll
        for (int k = 0; k < SWP; ++k) {
            if (FP8)
                dst[k] = (uint32_t)(rl * D + ((D == 128 ? ((cc ^ rl ^ (RPI * k)) & 7) : cc) << 4));
            else
                dst[k] = (uint32_t)(rl * 128 + (cc >> 3) * (UNIT * 128) + ((((cc & 7) ^ rl ^ (RPI * k)) & 7) << 4));
        }
    }
};

// Stage one unit (16 keys of K and of V) with 16-byte cp.async copies, written
// in the 128-byte-swizzled layout the ldmatrix reads expect: 16-byte chunk c of
// row r of a 64-column box sits at r * 128 + ((c ^ (r & 7)) * 16).  Lanes
// 0-15 / 16-31 copy two consecutive 256-byte rows per instruction (coalesced).
// Rows past the sequence end are not copied; their V rows are zeroed (their
// slots may hold anything and 0 * NaN = NaN), their K rows are masked later.
// Every call commits exactly one cp.async group (possibly empty).
template <int D, bool FP8, bool SWAP, bool APPEND>
__device__ __forceinline__ void issue_unit(const Params& p, const UnitIter& it, int phys, uint8_t* stage,
                                           int* phys_slot, int lane, uint64_t policy, const CopyLanes<D, FP8>& cl) {
    using C = Cfg<D, FP8, SWAP>;
    constexpr int CH = D / 8;  // 16-byte chunks per row (bf16)
    const int j = (it.u - it.seg.start) >> it.seg.sh.nrb_shift;  // key block within the sequence
    const int tok0 = j * UNIT;
    const int page = tok0 >> p.ps_shift;
    const int sub = (tok0 - (page << p.ps_shift)) / UNIT;
    if (phys < 0 || phys >= p.num_pages) {
        if (lane == 0) {
            report(p.status, PA_ERR_BAD_PAGE);
            *phys_slot = -1;
        }
    } else {
        if (lane == 0) *phys_slot = phys;
        const size_t row = (size_t)(phys * p.Hkv + it.seg.g) * p.page_size + sub * UNIT;
        const int valid = min(UNIT, it.seg.sh.len - tok0);
        const uint32_t sbase = smem_u32(stage);
        if constexpr (FP8) {
            // K: 16 rows of D bytes, 16-byte chunk c of row r at r * D + ((c ^ swz(r)) << 4);
            // V (transposed in the page): D rows of this unit's 16 key bytes, row d at d * 16
            constexpr int KCH = D / 16;
            constexpr int NCH = UNIT * KCH + D;
            const char* ksrc = reinterpret_cast<const char*>(p.k_pool) + row * D;
            const char* vsrc = reinterpret_cast<const char*>(p.v_pool) +
                               (size_t)(phys * p.Hkv + it.seg.g) * D * p.page_size + sub * UNIT;
            if (valid == UNIT) {
                // every K row is valid: no per-row test, addresses from cl
                using CL = CopyLanes<D, true>;
                const char* ks = ksrc + cl.src;
#pragma unroll
                for (int jj = 0; jj < CL::STEPS; ++jj)
                    cp_async_16(sbase + jj * CL::RPI * D + cl.dst[jj % CL::SWP], ks + jj * CL::RPI * D, policy);
                const char* vs = vsrc + (size_t)lane * p.page_size;
                const size_t vstep = (size_t)32 * p.page_size;
#pragma unroll
                for (int jj = 0; jj < D / 32; ++jj)
                    cp_async_16(sbase + C::UNIT_BYTES + (jj * 32 + lane) * 16, vs + jj * vstep, policy);
                cp_async_commit();
                return;
            }
#pragma unroll
            for (int i = 0; i < NCH / 32; ++i) {
                const int q = i * 32 + lane;
                if (q < UNIT * KCH) {
                    const int r = q / KCH, c = q - r * KCH;
                    const int sw = D == 128 ? (r & 7) : 0;
                    if (r < valid) cp_async_16(sbase + r * D + ((c ^ sw) << 4), ksrc + r * D + c * 16, policy);
                } else {
                    const int d = q - UNIT * KCH;  // keys past the end are cleared when the values are read
                    cp_async_16(sbase + C::UNIT_BYTES + d * 16, vsrc + (size_t)d * p.page_size, policy);
                }
            }
        } else {
            const char* ksrc = reinterpret_cast<const char*>(p.k_pool + row * D);
            const char* vsrc = reinterpret_cast<const char*>(p.v_pool + row * D);
            // append: rows r >= nf of the unit are the query tokens' own K/V (new token r - nf of
            // the sequence), not yet in the pool; that unit (one per sequence and head) is staged
            // by a second copy loop that takes them from k_new / v_new
            const int nf = APPEND ? it.seg.sh.len - it.seg.sh.qlen - tok0 : UNIT;
            if (valid == UNIT && nf >= UNIT) {
                // every row of the unit is in the pool: no per-row test, addresses from cl
                using CL = CopyLanes<D, false>;
                const char* ks = ksrc + cl.src;
                const char* vs = vsrc + cl.src;
#pragma unroll
                for (int jj = 0; jj < CL::STEPS; ++jj) {
                    const uint32_t d = sbase + cl.dst[jj % CL::SWP] + jj * CL::RPI * 128;
                    cp_async_16(d, ks + jj * CL::RPI * D * 2, policy);
                    cp_async_16(d + C::UNIT_BYTES, vs + jj * CL::RPI * D * 2, policy);
                }
            } else if (APPEND && nf < UNIT) {
                const size_t nrow = q_row(p, it.seg.b) * p.Hkv + it.seg.g;  // new token 0, head g
                const char* knew = reinterpret_cast<const char*>(p.k_new + nrow * D);
                const char* vnew = reinterpret_cast<const char*>(p.v_new + nrow * D);
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    const int q = i * 32 + lane;
                    const int t = q / (UNIT * CH);  // 0 = K, 1 = V
                    const int qq = q - t * UNIT * CH;
                    const int r = qq / CH;
                    const int cc = qq - r * CH;
                    const uint32_t dst = sbase + t * C::UNIT_BYTES + (cc >> 3) * C::BOX_BYTES + r * 128 +
                                         (((cc & 7) ^ (r & 7)) << 4);
                    if (r < valid) {
                        const char* src = r >= nf ? (t ? vnew : knew) + (size_t)(r - nf) * p.Hkv * D * 2 + cc * 16
                                                  : (t ? vsrc : ksrc) + r * D * 2 + cc * 16;
                        cp_async_16(dst, src, policy);
                    } else if (t == 1) {
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    const int q = i * 32 + lane;
                    const int t = q / (UNIT * CH);  // 0 = K, 1 = V
                    const int qq = q - t * UNIT * CH;
                    const int r = qq / CH;
                    const int cc = qq - r * CH;
                    const uint32_t dst = sbase + t * C::UNIT_BYTES + (cc >> 3) * C::BOX_BYTES + r * 128 +
                                         (((cc & 7) ^ (r & 7)) << 4);
                    if (r < valid) {
                        cp_async_16(dst, (t ? vsrc : ksrc) + r * D * 2 + cc * 16, policy);
                    } else if (t == 1) {
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
                    }
                }
            }
        }
    }
    cp_async_commit();
}

// fp16 tensor-core product (FP8 variant: e4m3 codes are exact in fp16)
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// four e4m3 codes (bytes 0 .. 3 of w) -> two fp16 pairs: lo = codes 0, 1 and hi = codes 2, 3
// (low half first); exact.  One conversion instruction per pair, reading the 16-bit halves
// of w in place (a helper that returns the halves separately costs two byte permutes more
// per pair to split and repack them).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 cl, ch;\n\tmov.b32 {cl, ch}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, cl;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, ch;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// FP8 variant: in the unit holding a sequence's last key (fewer than 16 valid
// keys), clear the staged value codes of the keys past the end: their slots
// may hold any code, NaN included, and 0 * NaN = NaN.  The transposed value
// block is D rows of 16 key bytes; word w of a row holds keys 4w .. 4w + 3.
// Other units are left alone (valid >= 16: nothing to clear).
template <int D>
__device__ __forceinline__ void clear_codes_past_end(uint32_t vb, int valid, int lane) {
    if (valid >= UNIT) return;
    for (int i = lane; i < D * 4; i += 32) {
        const int w = i & 3;
        uint32_t keep = 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (w * 4 + b < valid) keep |= 0xFFu << (8 * b);
        if (keep != 0xFFFFFFFFu) {
            const uint32_t addr = vb + (i >> 2) * 16 + w * 4;
            uint32_t x;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(addr));
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(x & keep) : "memory");
        }
    }
    __syncwarp();
}

// 8x8 b16 transpose across the warp (lane holds row lane/4, columns 2 (lane%4) + {0,1})
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// How the units [0, T) of a launch are cut into chunks, one per CTA of a grid
// of G; the decode and the merge kernel derive it from the same T and G.
// Chunk c owns workspace slots c + (segment index).  (Cutting the last part
// into small chunks that idle CTAs take from a counter was measured: the
// CTAs' finishing spread is about 10 %, and the extra partials cost the merge
// more than the balance gained.)
struct Split {
    int T, S;
    __device__ __forceinline__ Split(int T_, int G, int min_chunk) : T(T_), S(max(min_chunk, (T_ + G - 1) / G)) {}
    __device__ __forceinline__ int chunk_of(int u) const { return u / S; }
};

// Swapped-operand variant (SWAP, for at most 8 query rows per segment, e.g.
// decode with a GQA group of up to 8): the scores are computed transposed,
// S^T = K Q^T with the 16 keys of a unit as the mma's M and the 8 rows as its
// N, and the output as O^T = V^T P^T, P^T coming from the S^T accumulators by
// an 8x8 register transpose (movmatrix).  That is 16 mma per unit instead of
// 32 (the padded rows of a 16-row M are gone) and half the accumulator
// registers.  A lane's two softmax rows are 2 (lane & 3) and 2 (lane & 3) + 1.
//
// FP8 variant, key order inside a 16-key unit: score column c of n-tile t
// (the mma's n index) is key ((c >> 1) << 2) + 2t + (c & 1), so the four keys a
// lane feeds to P.V are four consecutive keys, i.e. one 32-bit word of a
// transposed value row.  The head dimension is likewise permuted: k-index
// (lane & 3) * 2 + j of k-step kk reads dimension (lane & 3) * D/4 + 4 kk + j,
// and k-index 8 + (lane & 3) * 2 + j reads that + 2, so each lane's K bytes
// and Q values are one contiguous run of D/4 dimensions.
//
// APPEND (bf16 pools): the query tokens' own K/V rows are not in the pool yet;
// the unit holding them stages them from k_new / v_new, and one warp per
// (sequence, KV head) writes them into their pool slots after using them.
//
// SW selects the operand order: 0 = plain (query rows as M), 1 = swapped for
// every segment, 2 = chosen per segment (swapped when the segment has at most
// 8 rows), for a call that mixes one-row entries with longer query blocks
// (the decode rows of a mixed serving step).
// Per-CTA scalars of the decode in shared memory (one set per virtual CTA).
template <int D, bool FP8, int SW>
struct DecShared {
    int s_phys[W][Cfg<D, FP8, SW == 1>::DEPTH];  // page of each staged unit (-1: bad entry)
    float s_m[W][RB], s_l[W][RB], s_M[RB], s_L[RB];
    int s_plan[8];
};

// Barrier over the W warps of one (virtual) CTA.
__device__ __forceinline__ void vsync(int bar_id) {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(W * 32) : "memory");
}

// The split-K decode of one CTA of a grid of nvcta, as W warps (tid 0 .. 32 W - 1)
// with their own shared memory (`smem`, 1024-byte aligned, Cfg::SMEM_BYTES) and
// named barrier `bar_id`.  The decode kernel runs it once per CTA; the mixed-step
// kernel runs two of these "virtual CTAs" per CTA, one per warpgroup.
template <int D, bool FP8, int SW, bool APPEND>
__device__ __forceinline__ void decode_body(const Params& p, const int vcta, const int nvcta, const int tid,
                                            const int bar_id, uint8_t* smem, DecShared<D, FP8, SW>& ds) {
    constexpr bool SWAP = SW == 1;
    static_assert(SW >= 0 && SW <= 2 && !(FP8 && SW == 2), "operand order");
    using C = Cfg<D, FP8, SWAP>;
    constexpr int DEPTH = C::DEPTH;
    constexpr int KSTEPS = D / 16;
    constexpr int NT = D / 8;  // n-tiles of O

    uint8_t* stages = smem;
    float* merge_o = reinterpret_cast<float*>(smem + C::STAGES_BYTES);
    auto& s_phys = ds.s_phys;
    auto& s_m = ds.s_m;
    auto& s_l = ds.s_l;
    auto& s_M = ds.s_M;
    auto& s_L = ds.s_L;
    auto& s_plan = ds.s_plan;

    const int warp = tid >> 5, lane = tid & 31;
    // Launched as a programmatic dependent: until pdl_wait() below, the previous kernel
    // of the stream may still run (the writeback of the newest K/V rows lets its
    // dependents start at once).  Before the wait the kernel reads only seq_lens, cu_q
    // and block_table, which that kernel does not write, and writes nothing, so the
    // plan and the first block-table lookups overlap it.

    // ---- plan: total units T
    if (warp == 0) {
        int T = 0;
        for (int b0 = 0; b0 < p.batch; b0 += 32) {
            const int b = b0 + lane;
            T += warp_sum_int(b < p.batch ? seq_units(p, seq_shape(p, b)) : 0);
        }
        if (lane == 0) s_plan[0] = T;
    }
    vsync(bar_id);
    // ---- split: CTA c owns the equal range [c S, (c + 1) S) of the units
    const Split sp(s_plan[0], nvcta, p.min_chunk);
    const int U0 = vcta * sp.S;  // grid * chunk < 2^31 is checked on the host
    const int U1 = min(sp.T, U0 + sp.S);
    const bool has_work = U0 < U1;

    const uint64_t policy = policy_evict_first();
    uint8_t* my_stages = stages + warp * DEPTH * C::STAGE_BYTES;
    const CopyLanes<D, FP8> cl(lane);

    // per-lane ldmatrix geometry (see the fragment layouts of mma.m16n8k16)
    const int mi = lane >> 3, ri = lane & 7;
    const int k_key = ((mi >> 1) << 3) + ri;  // K: matrices (keys 0-7|8-15) x (d lo|hi)
    const int k_dsel = mi & 1;
    const int v_key = ((mi & 1) << 3) + ri;   // V (trans): matrices (keys lo|hi) x (d lo|hi)
    const int v_dsel = mi >> 1;
    const int qr = lane >> 2;       // row group of this lane in mma fragments
    const int qc = (lane & 3) * 2;  // column pair of this lane
    // this lane's ldmatrix address within a 64-column box for 16-byte chunk 2 k + dsel
    // (k = 0 .. 3) of its row: A = (v_key, v_dsel), B = (k_key, k_dsel); chunk 2 (k + 4) + dsel
    // is the same offset in the next box
    uint32_t offA[4], offB[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        offA[k] = (uint32_t)(v_key * 128 + (((2 * k + v_dsel) ^ (v_key & 7)) << 4));
        offB[k] = (uint32_t)(k_key * 128 + (((2 * k + k_dsel) ^ (k_key & 7)) << 4));
    }

    const int cidx = vcta;  // this range's chunk
    Seg seg0;
    UnitIter it;
    int phys0 = -1;  // page of this warp's first unit
    if (has_work) {
        // segment holding U0
        if (warp == 0) {
            int sb = -1, sP = 0, P = 0;
            for (int b0 = 0; b0 < p.batch && sb < 0; b0 += 32) {
                const int b = b0 + lane;
                const int n = (b < p.batch) ? seq_units(p, seq_shape(p, b)) : 0;
                const int incl = warp_incl_scan(n);
                const int tot = __shfl_sync(0xffffffffu, incl, 31);
                if (U0 < P + tot) {
                    const unsigned hit = __ballot_sync(0xffffffffu, P + incl > U0);
                    const int l = __ffs(hit) - 1;
                    sb = b0 + l;
                    sP = P + __shfl_sync(0xffffffffu, incl - n, l);
                }
                P += tot;
            }
            if (lane == 0) {
                s_plan[4] = sb;
                s_plan[5] = sP;
            }
        }
        vsync(bar_id);
        seg_set_seq(seg0, p, s_plan[4]);
        const int idx = (U0 - s_plan[5]) / seg0.n;  // (g, sb) index within sequence b
        seg0.g = idx / seg0.sh.SB;
        seg0.sb = idx - seg0.g * seg0.sh.SB;
        seg0.start = s_plan[5] + idx * seg0.n;
        seg0.end = seg0.start + seg0.n;

        it.seg = seg0;
        it.U1 = U1;
        it.pe = min(U1, seg0.end);
        it.u = U0 + warp;
        it.done = false;
        it.pc_base = -1;
        it.pc_phys = -1;
        it.norm(p, warp);
        if (!it.done) phys0 = unit_page(p, it, lane);
    }

    // the previous kernel's writes (K/V rows, possibly q) are visible from here on
    pdl_wait();

    if (warp == 0) {
        // first unit of each sequence, for the merge kernel
        if (vcta == 0) {
            int T = 0;
            for (int b0 = 0; b0 < p.batch; b0 += 32) {
                const int b = b0 + lane;
                const int n = b < p.batch ? seq_units(p, seq_shape(p, b)) : 0;
                const int incl = warp_incl_scan(n);
                if (b < p.batch) p.seg_base[b] = T + incl - n;
                T += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) p.seg_base[p.batch] = T;
        }
        // empty sequences have a defined result: out = 0, lse = -inf
        for (int b = vcta; b < p.batch; b += nvcta) {
            const SeqShape sh = seq_shape(p, b);
            if (sh.qlen > 0 && sh.len == 0) {
                const size_t row0 = q_row(p, b) * p.Hq;
                for (int i = lane; i < sh.qlen * p.Hq * (D / 8); i += 32)
                    reinterpret_cast<uint4*>(p.out + row0 * D)[i] = make_uint4(0, 0, 0, 0);
                if (p.lse)
                    for (int i = lane; i < sh.qlen * p.Hq; i += 32) p.lse[row0 + i] = -INFINITY;
            }
        }
    }
    if (!has_work) return;

    // ---- prologue: fill this warp's pipeline, one cp.async group per stage (empty
    // groups once the warp runs out of units)
    uint32_t consumed = 0;
    for (int i = 0; i < DEPTH; ++i) {
        if (!it.done) {
            const int phys = i == 0 ? phys0 : unit_page(p, it, lane);
            issue_unit<D, FP8, SWAP, APPEND>(p, it, phys, my_stages + i * C::STAGE_BYTES, &s_phys[warp][i], lane, policy,
                                             cl);
            it.u += W;
            it.norm(p, warp);
        } else {
            cp_async_commit();
        }
    }

    Seg cs = seg0;
    int pa_ = U0;
    while (true) {
        const int pe = min(U1, cs.end);
        const int nrb = 1 << cs.sh.nrb_shift;
        const int rbase = (pa_ - cs.start) & (nrb - 1);  // row block of warp 0 in this piece
        const int wrb = (rbase + warp) & (nrb - 1);      // this warp's row block
        const int row_sb = cs.sb * cs.sh.RSB;             // first row of the segment
        const int rows_sb = min(cs.sh.RSB, cs.sh.qlen * p.group - row_sb);
        const int my_rows = max(0, min(cs.sh.R, rows_sb - wrb * cs.sh.R));
        const int qlast = cs.sh.len - cs.sh.qlen;  // position of query token 0
        // operand order of this piece (uniform over the CTA: every warp works on this segment)
        const bool swp = SW == 2 ? cs.sh.qlen * p.group <= 8 : SWAP;

        // Q fragments of this warp's rows (rows >= my_rows are zero) and the
        // number of keys each of the lane's two rows may see
        uint32_t qa[KSTEPS][4];
        int lim0 = cs.sh.len, lim1 = cs.sh.len, lim_all;
        // this lane's two softmax rows
        const int rA = swp ? (lane & 3) * 2 : qr, rB = swp ? rA + 1 : qr + 8;
        {
            const size_t qrow = q_row(p, cs.b);
            // rows whose q this lane loads: qr and qr + 8 (SWAP: only qr, as a column of Q^T)
            const bool r0ok = qr < my_rows, r8ok = !swp && qr + 8 < my_rows;
            const int f0 = row_sb + wrb * cs.sh.R + qr, f8 = f0 + 8;
            const int i0 = f0 / p.group, i8 = f8 / p.group;
            const int h0 = cs.g * p.group + (f0 - i0 * p.group), h8 = cs.g * p.group + (f8 - i8 * p.group);
            {
                const int fa = row_sb + wrb * cs.sh.R + rA, fb = row_sb + wrb * cs.sh.R + rB;
                if (rA < my_rows) lim0 = qlast + fa / p.group + 1;
                if (rB < my_rows) lim1 = qlast + fb / p.group + 1;
            }
            // units ending at or below every row's limit need no mask
            lim_all = __reduce_min_sync(0xffffffffu, min(lim0, lim1));
            const uint32_t* q0 = reinterpret_cast<const uint32_t*>(p.q + ((qrow + (r0ok ? i0 : 0)) * p.Hq + h0) * D);
            const uint32_t* q8 = reinterpret_cast<const uint32_t*>(p.q + ((qrow + (r8ok ? i8 : 0)) * p.Hq + h8) * D);
            if constexpr (FP8) {
                // fp16 fragments in the permuted dimension order (see above the kernel)
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int c = ((lane & 3) * (D / 4) + 4 * kk) >> 1;  // bf16 pair index
                    uint2 v0 = make_uint2(0u, 0u), v8 = make_uint2(0u, 0u);
                    if (r0ok) v0 = __ldg(reinterpret_cast<const uint2*>(q0 + c));
                    if (r8ok) v8 = __ldg(reinterpret_cast<const uint2*>(q8 + c));
                    const __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&v0.x);
                    const __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v0.y);
                    const __nv_bfloat162 e = *reinterpret_cast<__nv_bfloat162*>(&v8.x);
                    const __nv_bfloat162 f = *reinterpret_cast<__nv_bfloat162*>(&v8.y);
                    qa[kk][0] = pack_f16x2(__low2float(a), __high2float(a));
                    qa[kk][SWAP ? 1 : 2] = pack_f16x2(__low2float(b), __high2float(b));
                    if constexpr (!SWAP) {  // (no per-segment order for FP8)
                        qa[kk][1] = pack_f16x2(__low2float(e), __high2float(e));
                        qa[kk][3] = pack_f16x2(__low2float(f), __high2float(f));
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int c = (kk * 16 + qc) >> 1;
                    if (swp) {
                        qa[kk][0] = r0ok ? __ldg(q0 + c) : 0u;
                        qa[kk][1] = r0ok ? __ldg(q0 + c + 4) : 0u;
                    } else {
                        qa[kk][0] = r0ok ? __ldg(q0 + c) : 0u;
                        qa[kk][1] = r8ok ? __ldg(q8 + c) : 0u;
                        qa[kk][2] = r0ok ? __ldg(q0 + c + 4) : 0u;
                        qa[kk][3] = r8ok ? __ldg(q8 + c + 4) : 0u;
                    }
                }
            }
        }
        // score scale (log2 domain) and value scale of this KV head
        const float sl = FP8 ? p.scale_log2 * __ldg(p.k_scale + cs.g) : p.scale_log2;
        const float vsc = FP8 ? __ldg(p.v_scale + cs.g) : 1.f;
        float o[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        for (int u = pa_ + warp; u < pe; u += W) {
            const int st = consumed % DEPTH;
            cp_async_wait_group<DEPTH - 1>();  // this unit's group (DEPTH - 1 younger ones may fly)
            __syncwarp();
            const int phys = s_phys[warp][st];
            uint8_t* sk = my_stages + st * C::STAGE_BYTES;
            uint8_t* sv = sk + C::UNIT_BYTES;
            if (swp && phys >= 0) {
                const int tok0 = ((u - cs.start) >> cs.sh.nrb_shift) * UNIT;
                const int vis0 = lim0 - tok0, vis1 = lim1 - tok0;  // keys of this unit rows rA / rB see
                const uint32_t kb = smem_u32(sk), vb = smem_u32(sv);
                // S^T = K Q^T (16 keys x 8 rows), two accumulator chains (even / odd k-steps)
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                // keys of this lane's accumulator rows (FP8: permuted, see above the kernel)
                const int keyA = FP8 ? ((qr >> 1) << 2) + (qr & 1) : qr;
                const int keyB = FP8 ? keyA + 2 : qr + 8;
                if constexpr (FP8) {
                    uint32_t w0[D / 16], w1[D / 16];
#pragma unroll
                    for (int m = 0; m < D / 64; ++m) {
                        const int c = (lane & 3) * (D / 64) + m;
                        const int swa = D == 128 ? (keyA & 7) : 0, swb = D == 128 ? (keyB & 7) : 0;
                        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(w0[4 * m]), "=r"(w0[4 * m + 1]), "=r"(w0[4 * m + 2]), "=r"(w0[4 * m + 3])
                                     : "r"(kb + keyA * D + ((c ^ swa) << 4)));
                        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(w1[4 * m]), "=r"(w1[4 * m + 1]), "=r"(w1[4 * m + 2]), "=r"(w1[4 * m + 3])
                                     : "r"(kb + keyB * D + ((c ^ swb) << 4)));
                    }
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        uint32_t a[4];
                        e4m3x4_to_f16x2x2(w0[kk], a[0], a[2]);
                        e4m3x4_to_f16x2x2(w1[kk], a[1], a[3]);
                        const uint32_t (&qb)[4] = qa[kk];
                        mma_16816_f16((kk & 1) ? sb : sa, a, qb[0], qb[1]);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        const uint32_t addr = kb + (kk >> 2) * C::BOX_BYTES + offA[kk & 3];
                        uint32_t a[4];
                        ldsm_x4(addr, a[0], a[1], a[2], a[3]);
                        mma_16816((kk & 1) ? sb : sa, a, qa[kk][0], qa[kk][1]);
                    }
                }
                // scale, mask: element 0 / 1 = (keyA, rows rA / rB), 2 / 3 = (keyB, rows rA / rB)
                float x0 = (sa[0] + sb[0]) * sl, x1 = (sa[1] + sb[1]) * sl;
                float x2 = (sa[2] + sb[2]) * sl, x3 = (sa[3] + sb[3]) * sl;
                if (tok0 + UNIT > lim_all) {
                    x0 = keyA < vis0 ? x0 : -INFINITY;
                    x1 = keyA < vis1 ? x1 : -INFINITY;
                    x2 = keyB < vis0 ? x2 : -INFINITY;
                    x3 = keyB < vis1 ? x3 : -INFINITY;
                }
                float rm0 = fmaxf(x0, x2), rm1 = fmaxf(x1, x3);
#pragma unroll
                for (int o_ = 4; o_ < 32; o_ <<= 1) {
                    rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, o_));
                    rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, o_));
                }
                const float mn0 = rm0 > m0 + kDecTau ? rm0 : m0, mn1 = rm1 > m1 + kDecTau ? rm1 : m1;
                const float mr0 = mn0 == -INFINITY ? 0.f : mn0, mr1 = mn1 == -INFINITY ? 0.f : mn1;
                const float a0 = ex2(m0 - mr0), a1 = ex2(m1 - mr1);
                m0 = mn0;
                m1 = mn1;
                const float p0 = ex2(x0 - mr0), p2 = ex2(x2 - mr0), p1 = ex2(x1 - mr1), p3 = ex2(x3 - mr1);
                l0 = l0 * a0 + (p0 + p2);
                l1 = l1 * a1 + (p1 + p3);
                if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                    for (int n = 0; n < D / 16; ++n) {
                        o[n][0] *= a0;
                        o[n][1] *= a1;
                        o[n][2] *= a0;
                        o[n][3] *= a1;
                    }
                }
                // P^T (keys x rows) fragments: transpose the two 8x8 blocks of P
                const uint32_t b0 = movmatrix_trans(FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1));
                const uint32_t b1 = movmatrix_trans(FP8 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3));
                // O^T += V^T P^T, 16 value dimensions per mma
                if constexpr (FP8) {
                    clear_codes_past_end<D>(vb, cs.sh.len - tok0, lane);
#pragma unroll
                    for (int n = 0; n < D / 16; ++n) {
                        uint32_t wl, wh;
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wl) : "r"(vb + (n * 16 + qr) * 16 + (lane & 3) * 4));
                        asm volatile("ld.shared.u32 %0, [%1];"
                                     : "=r"(wh)
                                     : "r"(vb + (n * 16 + 8 + qr) * 16 + (lane & 3) * 4));
                        uint32_t a[4];
                        e4m3x4_to_f16x2x2(wl, a[0], a[2]);
                        e4m3x4_to_f16x2x2(wh, a[1], a[3]);
                        mma_16816_f16(o[n], a, b0, b1);
                    }
                } else {
#pragma unroll
                    for (int n = 0; n < D / 16; ++n) {
                        const uint32_t addr = vb + (n >> 2) * C::BOX_BYTES + offB[n & 3];
                        uint32_t a[4];
                        ldsm_x4_trans(addr, a[0], a[1], a[2], a[3]);
                        mma_16816(o[n], a, b0, b1);
                    }
                }
            } else if (!swp && phys >= 0) {
                const int tok0 = ((u - cs.start) >> cs.sh.nrb_shift) * UNIT;
                const int vis0 = lim0 - tok0, vis1 = lim1 - tok0;  // keys of this unit each row sees
                const uint32_t kb = smem_u32(sk), vb = smem_u32(sv);
                // S = Q K^T  (16 heads x 16 keys)
                // two independent accumulator chains (even / odd k-steps) halve the
                // dependent mma latency; summed below
                float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                if constexpr (FP8) {
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int krow = ((qr >> 1) << 2) + 2 * t + (qr & 1);  // key of n-tile t, column qr
                        uint32_t w[D / 16];  // this lane's D/4 bytes of that key row
#pragma unroll
                        for (int m = 0; m < D / 64; ++m) {
                            const int c = (lane & 3) * (D / 64) + m;
                            const int sw = D == 128 ? (krow & 7) : 0;
                            uint32_t r0, r1, r2, r3;
                            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                         : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                                         : "r"(kb + krow * D + ((c ^ sw) << 4)));
                            w[4 * m] = r0;
                            w[4 * m + 1] = r1;
                            w[4 * m + 2] = r2;
                            w[4 * m + 3] = r3;
                        }
#pragma unroll
                        for (int kk = 0; kk < KSTEPS; ++kk) {
                            uint32_t b0, b1;
                            e4m3x4_to_f16x2x2(w[kk], b0, b1);
                            mma_16816_f16((kk & 1) ? s2[t] : s[t], qa[kk], b0, b1);
                        }
                    }
                } else {
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const uint32_t addr = kb + (kk >> 2) * C::BOX_BYTES + offB[kk & 3];
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    if (kk & 1) {
                        mma_16816(s2[0], qa[kk], b0, b1);
                        mma_16816(s2[1], qa[kk], b2, b3);
                    } else {
                        mma_16816(s[0], qa[kk], b0, b1);
                        mma_16816(s[1], qa[kk], b2, b3);
                    }
                }
                }
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[j][e] += s2[j][e];
                // scale to log2 domain, mask keys past the sequence end or the row's position
                float x[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[j][e] = s[j][e] * sl;
                if (tok0 + UNIT > lim_all) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int key = FP8 ? (lane & 3) * 4 + 2 * j + (e & 1) : j * 8 + qc + (e & 1);
                            if (key >= ((e & 2) ? vis1 : vis0)) x[j][e] = -INFINITY;
                        }
                    }
                }
                float rm0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
                float rm1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
                rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 1));
                rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 2));
                rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 1));
                rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 2));
                const float mn0 = rm0 > m0 + kDecTau ? rm0 : m0, mn1 = rm1 > m1 + kDecTau ? rm1 : m1;
                // a row with no visible key yet keeps m = -inf; measure from 0 then so
                // that nothing computes -inf - (-inf)
                const float mr0 = mn0 == -INFINITY ? 0.f : mn0, mr1 = mn1 == -INFINITY ? 0.f : mn1;
                const float a0 = ex2(m0 - mr0), a1 = ex2(m1 - mr1);  // 0 when m was -inf
                m0 = mn0;
                m1 = mn1;
                float pr[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    pr[j][0] = ex2(x[j][0] - mr0);
                    pr[j][1] = ex2(x[j][1] - mr0);
                    pr[j][2] = ex2(x[j][2] - mr1);
                    pr[j][3] = ex2(x[j][3] - mr1);
                }
                l0 = l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
                l1 = l1 * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
                if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        o[n][0] *= a0;
                        o[n][1] *= a0;
                        o[n][2] *= a1;
                        o[n][3] *= a1;
                    }
                }
                uint32_t pa[4];
                if constexpr (FP8) {
                    pa[0] = pack_f16x2(pr[0][0], pr[0][1]);
                    pa[1] = pack_f16x2(pr[0][2], pr[0][3]);
                    pa[2] = pack_f16x2(pr[1][0], pr[1][1]);
                    pa[3] = pack_f16x2(pr[1][2], pr[1][3]);
                    // O += P V: value row d of the transposed unit holds the 16 keys' codes;
                    // this lane's keys (lane & 3) * 4 .. + 3 are one word.
                    clear_codes_past_end<D>(vb, cs.sh.len - tok0, lane);
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        uint32_t w;
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(vb + (n * 8 + qr) * 16 + (lane & 3) * 4));
                        uint32_t b0, b1;
                        e4m3x4_to_f16x2x2(w, b0, b1);
                        mma_16816_f16(o[n], pa, b0, b1);
                    }
                } else {
                pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
                pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
                pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
                pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
                // O += P V
#pragma unroll
                for (int jj = 0; jj < D / 16; ++jj) {
                    const uint32_t addr = vb + (jj >> 2) * C::BOX_BYTES + offA[jj & 3];
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(addr, b0, b1, b2, b3);
                    mma_16816(o[2 * jj], pa, b0, b1);
                    mma_16816(o[2 * jj + 1], pa, b2, b3);
                }
                }
            }
            if constexpr (APPEND) {
                // append: the warp that staged this unit for segment 0 and row block 0 (exactly one
                // per key block and KV head) writes its new rows from shared memory to their slots
                if (phys >= 0 && cs.sb == 0 && wrb == 0 &&
                    ((u - cs.start) >> cs.sh.nrb_shift) * UNIT + UNIT > cs.sh.len - cs.sh.qlen) {
                    constexpr int CH = D / 8;  // 16-byte chunks per row
                    const int tok0 = ((u - cs.start) >> cs.sh.nrb_shift) * UNIT;
                    const int r1 = min(UNIT, cs.sh.len - tok0);
                    if (lane < 2 * CH) {
                        const int cc = lane % CH;
                        const bool isv = lane >= CH;
                        const size_t row0 = ((size_t)phys * p.Hkv + cs.g) * p.page_size + (tok0 & (p.page_size - 1));
                        for (int r = max(0, cs.sh.len - cs.sh.qlen - tok0); r < r1; ++r) {
                            uint4 v;
                            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                         : "r"(smem_u32(isv ? sv : sk) + (cc >> 3) * C::BOX_BYTES + r * 128 +
                                               (((cc & 7) ^ (r & 7)) << 4)));
                            *reinterpret_cast<uint4*>((isv ? p.v_pool_w : p.k_pool_w) + (row0 + r) * D + cc * 8) = v;
                        }
                    }
                }
            }
            __syncwarp();  // every lane is done reading this stage
            ++consumed;
            if (!it.done) {
                const int phys_next = unit_page(p, it, lane);
                issue_unit<D, FP8, SWAP, APPEND>(p, it, phys_next, my_stages + st * C::STAGE_BYTES,
                                                 &s_phys[warp][st], lane, policy, cl);
                it.u += W;
                it.norm(p, warp);
            } else {
                cp_async_commit();
            }
        }

        // ---- merge the states of the warps that hold the same row block (fixed order)
        // (a row's partial sums are spread over the lanes that hold its other keys)
        if (swp) {
#pragma unroll
            for (int o_ = 4; o_ < 32; o_ <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
            }
        } else {
#pragma unroll
            for (int o_ = 1; o_ < 4; o_ <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
            }
        }
        const bool row_owner = swp ? (lane >> 2) == 0 : (lane & 3) == 0;
        if (row_owner) {
            s_m[warp][rA] = m0;
            s_l[warp][rA] = l0;
            s_m[warp][rB] = m1;
            s_l[warp][rB] = l1;
        }
        vsync(bar_id);
        const int c0 = sp.chunk_of(cs.start), c1 = sp.chunk_of(cs.end - 1);
        const int sid = (cs.b * p.Hkv + cs.g) * p.SBmax + cs.sb;
        const bool single = (c0 == c1);
        const size_t orow = q_row(p, cs.b);
        for (int r = 0; r < nrb; ++r) {
            const int wfirst = (r - rbase) & (nrb - 1);  // lowest warp holding row block r
            if (wrb == r) {
                float M0 = -INFINITY, M1 = -INFINITY;
                for (int w = wfirst; w < W; w += nrb) {
                    M0 = fmaxf(M0, s_m[w][rA]);
                    M1 = fmaxf(M1, s_m[w][rB]);
                }
                float L0 = 0.f, L1 = 0.f;
                for (int w = wfirst; w < W; w += nrb) {
                    const float mw0 = s_m[w][rA], mw1 = s_m[w][rB];
                    L0 += (mw0 == -INFINITY) ? 0.f : s_l[w][rA] * ex2(mw0 - M0);
                    L1 += (mw1 == -INFINITY) ? 0.f : s_l[w][rB] * ex2(mw1 - M1);
                }
                const float sc0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - M0);
                const float sc1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - M1);
                if (warp == wfirst && row_owner) {
                    s_M[rA] = M0;
                    s_L[rA] = L0;
                    s_M[rB] = M1;
                    s_L[rB] = L1;
                }
                m0 = sc0;  // m and l are not needed any more: keep the scale factors
                m1 = sc1;
            }
            // warps add their rescaled O into one buffer in a fixed order
#pragma unroll 1
            for (int w = wfirst; w < W; w += nrb) {
                if (swp && warp == w) {
                    // O^T fragment: (d = 16 n + qr (+8), rows rA / rB)
#pragma unroll
                    for (int n = 0; n < D / 16; ++n) {
#pragma unroll
                        for (int hi = 0; hi < 2; ++hi) {
                            const int d = n * 16 + qr + 8 * hi;
                            float* pA = merge_o + rA * C::MSTRIDE + d;
                            float* pB = merge_o + rB * C::MSTRIDE + d;
                            float vA = o[n][2 * hi] * m0, vB = o[n][2 * hi + 1] * m1;
                            if (w > wfirst) {
                                vA += *pA;
                                vB += *pB;
                            }
                            *pA = vA;
                            *pB = vB;
                        }
                    }
                } else if (!swp && warp == w) {
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const int col = n * 8 + qc;
                        float2* a0 = reinterpret_cast<float2*>(merge_o + qr * C::MSTRIDE + col);
                        float2* a1 = reinterpret_cast<float2*>(merge_o + (qr + 8) * C::MSTRIDE + col);
                        float2 v0 = make_float2(o[n][0] * m0, o[n][1] * m0);
                        float2 v1 = make_float2(o[n][2] * m1, o[n][3] * m1);
                        if (w > wfirst) {
                            const float2 p0 = *a0, p1 = *a1;
                            v0.x += p0.x;
                            v0.y += p0.y;
                            v1.x += p1.x;
                            v1.y += p1.y;
                        }
                        *a0 = v0;
                        *a1 = v1;
                    }
                }
                vsync(bar_id);
            }
            const int nr = max(0, min(cs.sh.R, rows_sb - r * cs.sh.R));
            for (int idx = tid; idx < nr * (D / 4); idx += W * 32) {
                const int rr = idx / (D / 4);
                const int d4 = idx - rr * (D / 4);
                const float4 acc = *reinterpret_cast<const float4*>(merge_o + rr * C::MSTRIDE + d4 * 4);
                const float L = s_L[rr];
                const float inv = L > 0.f ? vsc / L : 0.f;  // the value scale folds in here
                if (single) {
                    const int f = row_sb + r * cs.sh.R + rr;
                    const int i = f / p.group;
                    const size_t orr = (orow + i) * p.Hq + cs.g * p.group + (f - i * p.group);
                    uint2 ob;
                    ob.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                    ob.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                    *reinterpret_cast<uint2*>(p.out + orr * D + d4 * 4) = ob;
                    if (p.lse != nullptr && d4 == 0) p.lse[orr] = L > 0.f ? (s_M[rr] + lg2(L)) * kLn2 : -INFINITY;
                } else {
                    const size_t srow = ((size_t)cidx + sid) * p.RS + r * RB + rr;
                    *reinterpret_cast<float4*>(p.ws_o + srow * D + d4 * 4) =
                        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                    if (d4 == 0) p.ws_lse[srow] = L > 0.f ? s_M[rr] + lg2(L) : -INFINITY;
                }
            }
            vsync(bar_id);  // the merge buffer and s_M / s_L are reused by the next row block
        }
        vsync(bar_id);  // merge buffers are reused by the next piece
        if (pe >= U1) break;
        pa_ = pe;
        seg_next(cs, p);
    }

    cp_async_wait_group<0>();  // never exit with a copy still landing in shared memory
}

template <int D, bool FP8, int SW, bool APPEND>
__global__ void __launch_bounds__(W * 32, ctas_per_sm<FP8, SW == 1>())
    decode_kernel(const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ DecShared<D, FP8, SW> ds;
    pdl_launch_dependents();  // the merge kernel may be scheduled (it waits for this grid)
    decode_body<D, FP8, SW, APPEND>(p, blockIdx.x, gridDim.x, threadIdx.x, 0, smem, ds);
}

// Merge of the split segments (the reduction step of Flash-Decoding):
//     lse = log sum_c exp(lse_c),   o = sum_c exp(lse_c - lse) o_c
// over the chunks c0 .. c1 of a segment, in chunk order.  Block (segment,
// row block), one thread per (row, 4 dimensions); each thread loads its
// row's partials eight chunks at a time and merges them with a running max.
// Launched right after the decode kernel as its programmatic dependent: the
// row geometry (from seq_lens / cu_q, which the decode does not write) is
// worked out while the decode finishes, then it waits for that grid, and
// lets the next kernel of the stream (the next step's decode, which reads
// only its unwritten inputs before its own wait) start its plan.
template <int D>
__global__ void __launch_bounds__(RB * D / 4) merge_kernel(const Params p) {
    if (p.reset_words != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        pdl_wait();  // the grid before (the mixed-step kernel) is done with them
        p.reset_words[0] = 0ull;
        p.reset_words[1] = 0ull;
    }
    const int sid = blockIdx.x;
    const int per_b = p.Hkv * p.SBmax;
    const int b = sid / per_b;
    const int g = (sid - b * per_b) / p.SBmax;
    const int sb = sid - b * per_b - g * p.SBmax;
    Seg s;
    seg_set_seq(s, p, b);
    if (s.n == 0 || sb >= s.sh.SB) return;
    const int r = blockIdx.y;
    if (r >= (1 << s.sh.nrb_shift)) return;
    const int rr = threadIdx.x / (D / 4), d4 = threadIdx.x - rr * (D / 4);
    const int row_sb = sb * s.sh.RSB;
    const int rows_sb = min(s.sh.RSB, s.sh.qlen * p.group - row_sb);
    if (rr >= min(s.sh.R, rows_sb - r * s.sh.R)) return;
    pdl_wait();
    pdl_launch_dependents();
    const int start = p.seg_base[b] + (g * s.sh.SB + sb) * s.n;
    const Split sp(p.seg_base[p.batch], p.G, p.min_chunk);
    const int c0 = sp.chunk_of(start), c1 = sp.chunk_of(start + s.n - 1);
    if (c0 == c1) return;  // one chunk held the whole segment and stored its rows
    const int rw = r * RB + rr;
    // one pass with a running max (rescaling when it grows), so that each partial's
    // lse and O loads are issued together
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int c = c0; c <= c1; ++c) {
        const size_t srow = ((size_t)c + sid) * p.RS + rw;
        const float lc = __ldcg(p.ws_lse + srow);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.ws_o + srow * D) + d4);
        const float mn = fmaxf(M, lc);
        const float sc = M == -INFINITY ? 0.f : ex2(M - mn);  // the state is all zero while M = -inf
        // a partial with no visible key has lse = -inf and O = 0
        const float wgt = lc == -INFINITY ? 0.f : ex2(lc - mn);
        L = L * sc + wgt;
        acc.x = acc.x * sc + wgt * v.x;
        acc.y = acc.y * sc + wgt * v.y;
        acc.z = acc.z * sc + wgt * v.z;
        acc.w = acc.w * sc + wgt * v.w;
        M = mn;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int f = row_sb + r * s.sh.R + rr;
    const int i = f / p.group;
    const size_t orr = (q_row(p, b) + i) * p.Hq + g * p.group + (f - i * p.group);
    uint2 ob;
    ob.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    ob.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.out + orr * D + d4 * 4) = ob;
    if (p.lse != nullptr && d4 == 0) p.lse[orr] = L > 0.f ? (M + lg2(L)) * kLn2 : -INFINITY;
}

// Workspace layout: [seg_base: batch + 1 int32][ws_lse: slots x RS f32][ws_o: slots x RS x D f32].
// Every part is written before it is read in a call: the workspace needs no initialisation.
struct WsLayout {
    size_t hdr, lse, o, total;
};

inline WsLayout ws_layout(int slots, int batch, int RS, int D) {
    WsLayout w;
    w.hdr = 0;
    w.lse = align_up((size_t)(batch + 1) * 4, 256);
    w.o = w.lse + align_up((size_t)slots * RS * 4, 256);
    w.total = w.o + (size_t)slots * RS * D * 4;
    return w;
}

// Largest segment count per (sequence, KV head) and rows per workspace slot
// over every q_len <= qmax (the device's seq_shape never exceeds them).
struct Bounds {
    int SBmax, RS;
};

inline Bounds bounds(int group, int qmax) {
    const int rows = group * qmax;
    Bounds bd;
    bd.SBmax = (rows + SBR - 1) / SBR;
    const int nrb = rows > SBR ? 4 : (rows + RB - 1) / RB;
    bd.RS = RB * (nrb <= 1 ? 1 : (nrb == 2 ? 2 : 4));
    return bd;
}

// Workspace slots: one per chunk (at most the largest grid), offset by the segment index.
inline int ws_slots(int sm_count, int segs) { return sm_count * kMaxCtasPerSM + segs; }

inline size_t ws_bytes(int sm_count, int batch, int num_q_heads, int num_kv_heads, int head_dim, int qmax) {
    const Bounds bd = bounds(num_q_heads / num_kv_heads, qmax);
    const int segs = batch * num_kv_heads * bd.SBmax;
    return ws_layout(ws_slots(sm_count, segs), batch, bd.RS, head_dim).total;
}

// A checked, ready-to-launch split-K decode (host side; decode.cu).
struct DecodeLaunch {
    Params prm;
    int grid;  // CTAs (or virtual CTAs) running the decode body; 0: nothing to launch
    long long segs;
    int nrb_max, head_dim, device, min_chunk, qmax;
    bool fp8, swap, mixed_order, app;
};

int prepare_decode(DecodeLaunch* L, void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                   const float* k_scale, const float* v_scale, const void* k_new, const void* v_new, int num_pages,
                   const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens, const int32_t* cu_q,
                   int total_q, int qmax, int qcap, int batch, int max_seq_len, int page_size, int num_q_heads,
                   int num_kv_heads, int head_dim, float softmax_scale, void* workspace, size_t workspace_bytes,
                   int32_t* status, bool per_segment, int grid_override);

// Launch the merge of the split segments of a prepared decode (after its decode grid).
int launch_merge(const DecodeLaunch& L, cudaStream_t st);

}  // namespace dec
}  // namespace pa
