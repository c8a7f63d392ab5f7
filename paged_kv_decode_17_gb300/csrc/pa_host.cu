// Host helpers of libpagedattn.so: status strings, device properties,
// tensor-map encoding through the driver entry point (no link-time
// dependency on libcuda).
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "pa_host.h"

namespace pa {

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices] = {};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
}

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

constexpr int kMaxKernelSlots = 32;
bool g_smem_set[kMaxDevices][kMaxKernelSlots] = {};

int encode_impl(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_elems, uint32_t box_cols,
                uint32_t box_rows, CUtensorMapSwizzle swz) {
    std::call_once(g_encode_once, load_encode);
    if (g_encode == nullptr) return PA_ERR_CUDA;
    cuuint64_t dims[2] = {row_elems, rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems) * 2u};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

int current_device(DeviceInfo* info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_have[dev]) {
            cudaDeviceProp p;
            if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return PA_ERR_CUDA;
            g_info[dev] = DeviceInfo{dev, p.multiProcessorCount, p.major, p.minor, p.sharedMemPerBlockOptin};
            g_have[dev] = true;
        }
        *info = g_info[dev];
    }
    if (info->major != 10 || info->minor != 3) return PA_ERR_ARCH;
    return PA_OK;
}

int current_context_id(unsigned long long* id) {
    std::call_once(g_ctx_once, load_ctx);
    if (g_ctx_current == nullptr || g_ctx_id == nullptr) return PA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PA_ERR_CUDA;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_elems, uint32_t box_cols,
                    uint32_t box_rows) {
    return encode_impl(map, base, rows, row_elems, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

int encode_rows_map_noswizzle(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_elems,
                              uint32_t box_cols, uint32_t box_rows) {
    return encode_impl(map, base, rows, row_elems, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

int encode_blocks_map(CUtensorMap* map, const void* base, uint64_t blocks) {
    std::call_once(g_encode_once, load_encode);
    if (g_encode == nullptr) return PA_ERR_CUDA;
    // a 16-row block of 128-column bf16 rows (4 KB) in the order [row half][column block][row][column]:
    // dimension 1 (rows) steps 256 bytes, dimension 2 (column block) 128, dimension 3 (row half) 2048
    cuuint64_t dims[5] = {64, 8, 2, 2, blocks};
    cuuint64_t strides[4] = {256, 128, 2048, 4096};
    cuuint32_t box[5] = {64, 8, 2, 2, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int encode_q_map(CUtensorMap* map, const void* q, int total_q, int Hq, int D) {
    std::call_once(g_encode_once, load_encode);
    if (g_encode == nullptr) return PA_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2u, (cuuint64_t)Hq * D * 2u};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int set_smem_limit_once(const void* kernel, int bytes, int device, int slot) {
    if (device < 0 || device >= kMaxDevices || slot < 0 || slot >= kMaxKernelSlots) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_set[device][slot]) return PA_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return PA_ERR_CUDA;
    g_smem_set[device][slot] = true;
    return PA_OK;
}

}  // namespace pa

extern "C" int pa_abi_version(void) { return 2; }

extern "C" const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_NULL: return "a required pointer is NULL";
        case PA_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA runtime/driver call or kernel launch failed";
        case PA_ERR_TIMEOUT: return "device: a prefill-kernel wait ran past its time limit";
        case PA_ERR_BAD_PAGE: return "device: block_table entry outside [0, num_pages)";
        case PA_ERR_BAD_LEN: return "device: sequence length / row count inconsistent";
        case PA_ERR_ARCH: return "current device is not an sm_103 GPU";
        case PA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the allocation-free decode holds (8 MiB)";
        default: return "unknown status";
    }
}
