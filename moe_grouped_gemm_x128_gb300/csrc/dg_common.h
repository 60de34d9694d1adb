// Internal host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg.h"

namespace dg {

constexpr int kQBlock = 128;  // K-group of the fine-grained scales and of one promotion step

// Per-device facts the launchers need, queried once per device.
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    unsigned int *status_word = nullptr;  // device address of the status word
};

// Fills `info` for the current device (cached).  Returns DG_ERR_CUDA if a
// runtime query failed and DG_ERR_UNSUPPORTED_DEVICE if the device is not
// compute capability 10.3.
dg_status_t current_device(DeviceInfo *info);

// Sets the maximum dynamic shared memory of `func` on the current device the
// first time it is asked for a given (device, func) pair.
dg_status_t ensure_smem_attr(const void *func, int smem_bytes);

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point.
dg_status_t encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base,
                              const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                              CUtensorMapSwizzle swizzle);

// The 256 x 256 tiles computed by a CTA pair (dg_gemm_pair.cu).  The
// contiguous layout's list of row pairs lives in shared memory, so the pair
// kernel takes at most this many 128-row blocks.
constexpr int kPairMaxRows = 1024;
bool pair_plan_ok(int layout, int M, int N, int K, int G, int num_sms);
int pair_smem_bytes();
int pair_num_tiles(int layout, int M, int N, int G);
dg_status_t launch_pair(int layout, const uint8_t *a, const float *sfa, const uint8_t *b, const float *sfb, uint16_t *d,
                        uint8_t *qout, float *sfo, const int32_t *meta, int M, int N, int K, int G,
                        int num_tiles_hint, void *stream, const DeviceInfo &info);

inline bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int ceil_div(int a, int b)
{
    return (a + b - 1) / b;
}

inline int round_up(int a, int b)
{
    return ceil_div(a, b) * b;
}

}  // namespace dg
