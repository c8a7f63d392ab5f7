// Host-side helpers shared by the launchers (argument checks, device
// properties, tensor-map encoding).  Internal to libpagedattn.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

struct DeviceInfo {
    int device;
    int sm_count;
    int major, minor;
    size_t max_smem_optin;
};

// Properties of the current device (cached per device).  Returns PA_OK,
// PA_ERR_CUDA or PA_ERR_ARCH (not an sm_103 GPU).
int current_device(DeviceInfo* info);

// Unique ID of the current CUDA context (a context created after a device
// reset gets a new one).  Returns PA_OK or PA_ERR_CUDA.
int current_context_id(unsigned long long* id);

// Encode a 2-D bf16 tensor map over `rows` rows of `row_elems` elements
// (row stride = row_elems * 2 bytes), box = box_cols x box_rows, 128-byte
// swizzle.  Returns PA_OK or PA_ERR_CUDA.
int encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_elems, uint32_t box_cols,
                    uint32_t box_rows);

// Same, without swizzle (plain row-major box).
int encode_rows_map_noswizzle(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_elems,
                              uint32_t box_cols, uint32_t box_rows);

// 3-D bf16 tensor map over q [total_q][Hq][D] with box {64, 1, 128} and
// 128-byte swizzle: one head's 128-row tile, 64 columns at a time.
// K or V pool at head_dim 128 as 16-row blocks: one box = one block (see pf::Cfg::BLK4).
int encode_blocks_map(CUtensorMap* map, const void* base, uint64_t blocks);
int encode_q_map(CUtensorMap* map, const void* q, int total_q, int Hq, int D);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks shared by every entry point.
inline int check_common_shapes(int page_size, int num_q_heads, int num_kv_heads, int head_dim) {
    if (head_dim != 64 && head_dim != 128) return PA_ERR_SHAPE;
    if (page_size < 16 || page_size > 256 || (page_size & (page_size - 1)) != 0) return PA_ERR_SHAPE;
    if (num_kv_heads < 1 || num_q_heads < num_kv_heads || num_q_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
    if (num_q_heads / num_kv_heads > 128) return PA_ERR_SHAPE;
    return PA_OK;
}

// Entries with q_len <= kDecodeMaxQ are served by the split-K decode kernel
// (also inside a mixed prefill + decode call); longer ones by the prefill kernel.
constexpr int kDecodeMaxQ = 8;

namespace dec {
// Split-K decode launcher (decode.cu).  cu_q == nullptr: one query row per
// sequence.  Otherwise the entries with 1 <= q_len <= qmax are served, q_len
// in (qmax, qcap] is reported as an error and longer entries are skipped.
// per_segment: choose the operand order per segment (one-row entries of a
// mixed call take the swapped-operand path even when qmax rows would not).
int launch_decode(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool, int num_pages,
                  const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                  const int32_t* cu_q, int total_q, int qmax, int qcap, int batch, int max_seq_len, int page_size,
                  int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale, void* workspace,
                  size_t workspace_bytes, int32_t* status, void* stream, bool per_segment = false);
}  // namespace dec

// Set the dynamic shared-memory limit of a kernel once per device.
int set_smem_limit_once(const void* kernel, int bytes, int device, int slot);

}  // namespace pa
