// Library-wide state and helpers: the device status word, per-device facts,
// status strings and tensor-map encoding.
#include <mutex>

#include "dg_common.h"
#include "dg_wait.cuh"

// Problems only the GPU can see (bad MoE metadata, pipeline timeouts) are
// OR-ed into this word by the kernels; dg_read_device_status reads and clears
// it.  Every kernel receives its device address as an argument.
__device__ unsigned int g_dg_status_word;

namespace dg {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxFuncs = 64;

struct DeviceSlot {
    bool ready = false;
    DeviceInfo info;
    const void *funcs[kMaxFuncs] = {};
    int func_smem[kMaxFuncs] = {};
    int nfuncs = 0;
};

std::mutex g_lock;
DeviceSlot g_slots[kMaxDevices];

}  // namespace

dg_status_t current_device(DeviceInfo *info)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return DG_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    DeviceSlot &slot = g_slots[dev];
    if (!slot.ready) {
        DeviceInfo d;
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return DG_ERR_CUDA;
        if (d.cc_major != 10 || d.cc_minor != 3) {
            *info = d;
            return DG_ERR_UNSUPPORTED_DEVICE;
        }
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dg_status_word) != cudaSuccess)
            return DG_ERR_CUDA;
        d.status_word = static_cast<unsigned int *>(p);
        slot.info = d;
        slot.ready = true;
    }
    *info = slot.info;
    return DG_OK;
}

dg_status_t ensure_smem_attr(const void *func, int smem_bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return DG_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    DeviceSlot &slot = g_slots[dev];
    for (int i = 0; i < slot.nfuncs; ++i)
        if (slot.funcs[i] == func && slot.func_smem[i] >= smem_bytes)
            return DG_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return DG_ERR_CUDA;
    for (int i = 0; i < slot.nfuncs; ++i)
        if (slot.funcs[i] == func) {
            slot.func_smem[i] = smem_bytes;
            return DG_OK;
        }
    if (slot.nfuncs < kMaxFuncs) {
        slot.funcs[slot.nfuncs] = func;
        slot.func_smem[slot.nfuncs] = smem_bytes;
        ++slot.nfuncs;
    }
    return DG_OK;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn resolve_encode()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

dg_status_t encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base,
                              const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                              CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = resolve_encode();
    if (!fn)
        return DG_ERR_CUDA;
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5];
    cuuint32_t estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i + 1 < rank)
            gstride[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void *>(base), gdim, gstride, bdim,
                    estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_ERR_CUDA;
}

}  // namespace dg

extern "C" const char *dg_status_string(dg_status_t status)
{
    switch (status) {
    case DG_OK:
        return "ok";
    case DG_ERR_INVALID_ARG:
        return "invalid argument (null pointer, non-positive size or unknown enum)";
    case DG_ERR_UNSUPPORTED_SHAPE:
        return "unsupported shape (K must be a multiple of 128, N a multiple of 8)";
    case DG_ERR_MISALIGNED:
        return "device pointer not 16-byte aligned";
    case DG_ERR_UNSUPPORTED_DEVICE:
        return "current device is not compute capability 10.3 (sm_103a)";
    case DG_ERR_CUDA:
        return "CUDA runtime or launch error";
    case DG_ERR_DEVICE_TIMEOUT:
        return "a kernel pipeline wait timed out; outputs are incomplete";
    }
    return "unknown status";
}

extern "C" dg_status_t dg_read_device_status(int *flags, void *stream)
{
    if (!flags)
        return DG_ERR_INVALID_ARG;
    dg::DeviceInfo info;
    dg_status_t st = dg::current_device(&info);
    if (st != DG_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, info.status_word, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(info.status_word, 0, sizeof(host), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DG_ERR_CUDA;
    *flags = static_cast<int>(host);
    return (host & DG_DEVFLAG_TIMEOUT) ? DG_ERR_DEVICE_TIMEOUT : DG_OK;
}

namespace dg {
namespace {

// One thread waits, with the GEMMs' bounded wait, on an mbarrier that nothing
// arrives on: the wait gives up after `limit` SM cycles, raises the CTA's
// abort flag and DG_DEVFLAG_TIMEOUT, and the kernel returns.  No copy, MMA or
// tensor memory is in flight, so nothing needs draining.
__global__ void __launch_bounds__(32) selftest_wait_timeout_kernel(long long limit, unsigned int *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_word;
    if (threadIdx.x != 0)
        return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbarrier_init();
    abort_word = 0;
    volatile uint32_t *abort_flag = &abort_word;
    // phase 0 never completes (its single arrival never comes), so the wait
    // returns false after `limit` cycles with DG_DEVFLAG_TIMEOUT raised
    (void)wait_phase(b, 0, abort_flag, status, limit);
}

}  // namespace
}  // namespace dg

extern "C" dg_status_t dg_selftest_wait_timeout(long long limit_cycles, void *stream)
{
    if (limit_cycles < 1000 || limit_cycles > dg::kWaitTimeoutCycles)
        return DG_ERR_INVALID_ARG;
    dg::DeviceInfo info;
    dg_status_t st = dg::current_device(&info);
    if (st != DG_OK)
        return st;
    dg::selftest_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles, info.status_word);
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}
