// FP8 quantisers: per-token 1x128 groups for activations and 128x128 blocks
// for weights ("DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库", 功能特色/细粒度缩放功能;
// 2kiu.com tutorial 4.4 精度控制与数值稳定性: scales from data statistics and
// saturation of out-of-range values).
//
// Rule per group: amax = max|x|, s = max(amax, 1e-4f) / 448 (IEEE fp32
// division), q = E4M3 RNE with saturation of fp32(x / s), the quotient
// rounded to nearest as IEEE division rounds it (computed by div2_rn: a
// correctly rounded reciprocal and two remainder corrections per value).
//
// The activation quantiser is HBM-bound on large inputs: 4 (or 2) bytes in
// and 1 + 4/128 bytes out per element.  One warp quantises one 128-value group
// with one 16-byte load per lane; a block of 8 warps covers 8 consecutive rows
// x GPW consecutive groups, so that the 8 scales of one group column land in
// one 32-byte sector.  Large inputs take GPW = 4 (four independent loads in
// flight per warp); small ones, latency-bound, take GPW = 1 so that the
// division chains spread over more warps.
#include "dg_common.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int kQuantWarps = 8;        // rows per block

__device__ __forceinline__ float4 load_group4(const float *x, size_t off)
{
    return __ldcs(reinterpret_cast<const float4 *>(x + off));
}

__device__ __forceinline__ float4 load_group4(const uint16_t *x, size_t off)
{
    uint2 u = __ldcs(reinterpret_cast<const uint2 *>(x + off));
    float4 f;
    f.x = __uint_as_float(u.x << 16);
    f.y = __uint_as_float(u.x & 0xFFFF0000u);
    f.z = __uint_as_float(u.y << 16);
    f.w = __uint_as_float(u.y & 0xFFFF0000u);
    return f;
}

template <typename T, int GPW>
__global__ void __launch_bounds__(kQuantWarps * 32) quant_act_1x128_kernel(const T *__restrict__ x,
                                                                          uint8_t *__restrict__ q,
                                                                          float *__restrict__ sfa, int M, int K,
                                                                          int ldsfa)
{
    const int KB = K / kQBlock;
    const int row_tiles = (M + kQuantWarps - 1) / kQuantWarps;
    const int col_tiles = (KB + GPW - 1) / GPW;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // a GEMM launched after this kernel may start its prologue now; it waits
    // for this grid's completion before reading q or sfa
    griddep_launch_dependents();
    for (int task = blockIdx.x; task < row_tiles * col_tiles; task += gridDim.x) {
        const int m = (task / col_tiles) * kQuantWarps + warp;
        const int kb0 = (task % col_tiles) * GPW;
        if (m >= M)
            continue;
        float4 v[GPW];
#pragma unroll
        for (int j = 0; j < GPW; ++j)
            if (kb0 + j < KB)
                v[j] = load_group4(x, static_cast<size_t>(m) * K + static_cast<size_t>(kb0 + j) * kQBlock + lane * 4);
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
            const int kb = kb0 + j;
            if (kb >= KB)
                break;
            float amax = fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w)));
            amax = warp_max(amax);
            const float s = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
            const float y = __frcp_rn(s);
            const float2 lo = div2_rn(make_float2(v[j].x, v[j].y), s, y);
            const float2 hi = div2_rn(make_float2(v[j].z, v[j].w), s, y);
            const uint32_t packed = e4m3x4(lo.x, lo.y, hi.x, hi.y);
            __stcs(reinterpret_cast<uint32_t *>(q + static_cast<size_t>(m) * K + static_cast<size_t>(kb) * kQBlock) +
                       lane,
                   packed);
            if (lane == 0)
                sfa[static_cast<size_t>(kb) * ldsfa + m] = s;
        }
    }
}

// One block per (matrix g, 128-row block nb, 128-column block kb): 256 threads
// hold the 16384 values in registers, reduce amax, then quantise.
__global__ void __launch_bounds__(256) quant_weight_128x128_kernel(const float *__restrict__ w,
                                                                   uint8_t *__restrict__ q,
                                                                   float *__restrict__ sfb, int N, int K)
{
    const int KB = K / kQBlock;
    const int NB = (N + kQBlock - 1) / kQBlock;
    const int kb = blockIdx.x % KB;
    const int nb = (blockIdx.x / KB) % NB;
    const int g = blockIdx.x / (KB * NB);
    const float *wg = w + static_cast<size_t>(g) * N * K;
    uint8_t *qg = q + static_cast<size_t>(g) * N * K;
    __shared__ float red[8];

    float4 v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e = i * 256 + threadIdx.x;
        const int n = nb * kQBlock + e / 32;
        const int k = kb * kQBlock + (e % 32) * 4;
        if (n < N) {
            v[i] = *reinterpret_cast<const float4 *>(wg + static_cast<size_t>(n) * K + k);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
    }
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        amax = fmaxf(amax, red[i]);
    const float s = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
    const float y = __frcp_rn(s);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e = i * 256 + threadIdx.x;
        const int n = nb * kQBlock + e / 32;
        const int k = kb * kQBlock + (e % 32) * 4;
        if (n < N) {
            const float2 lo = div2_rn(make_float2(v[i].x, v[i].y), s, y);
            const float2 hi = div2_rn(make_float2(v[i].z, v[i].w), s, y);
            *reinterpret_cast<uint32_t *>(qg + static_cast<size_t>(n) * K + k) = e4m3x4(lo.x, lo.y, hi.x, hi.y);
        }
    }
    if (threadIdx.x == 0)
        sfb[(static_cast<size_t>(g) * NB + nb) * KB + kb] = s;
}

// MX quantiser (OCP Microscaling v1.0 with E4M3 elements): per row and
// 32-wide block, e = floor(log2 amax) - 8 clamped to [-127, 127] (an all-zero
// or subnormal block takes -127), scale code e + 127, codes E4M3 RNE with
// saturation of x * 2^-e.  One warp quantises four blocks of one row (128
// values, one 16-byte load per lane); the eight lanes of a block reduce its
// amax with shuffles.  floor(log2 amax) is amax's exponent field; x * 2^-e
// is one multiplication by a power of two, exact unless the product is
// subnormal, where it is correctly rounded and then encodes to +-0.
__global__ void __launch_bounds__(256) quant_mx_1x32_kernel(const float *__restrict__ x, uint8_t *__restrict__ q,
                                                             uint8_t *__restrict__ sx, int R, int K)
{
    const int groups = K / 128;                   // 128-value groups per row
    const long long tasks = static_cast<long long>(R) * groups;
    const int lane = threadIdx.x & 31;
    for (long long task = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5); task < tasks;
         task += static_cast<long long>(gridDim.x) * 8) {
        const int r = static_cast<int>(task / groups);
        const int g = static_cast<int>(task % groups);
        const size_t off = static_cast<size_t>(r) * K + static_cast<size_t>(g) * 128 + lane * 4;
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(x + off));
        float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        // lanes 8b..8b+7 hold block b of the group
#pragma unroll
        for (int o = 4; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int expo = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);   // 0 for zero / subnormal
        int e = expo == 0 ? -127 : expo - 127 - 8;
        e = e < -127 ? -127 : (e > 127 ? 127 : e);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);      // 2^-e, a normal float
        const uint32_t packed = e4m3x4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
        __stcs(reinterpret_cast<uint32_t *>(q + off), packed);
        // the group's four scale codes as one word (byte j = block j), stored
        // chunk-major: word [g][r]
        const uint32_t code = static_cast<uint32_t>(e + 127);
        const uint32_t word = __shfl_sync(0xffffffffu, code, 0) | (__shfl_sync(0xffffffffu, code, 8) << 8) |
                              (__shfl_sync(0xffffffffu, code, 16) << 16) | (__shfl_sync(0xffffffffu, code, 24) << 24);
        if (lane == 0)
            reinterpret_cast<uint32_t *>(sx)[static_cast<size_t>(g) * R + r] = word;
    }
}

}  // namespace
}  // namespace dg

extern "C" dg_status_t dg_quant_act_1x128(const void *x, int x_dtype, uint8_t *q, float *sfa, int M, int K,
                                          void *stream)
{
    using namespace dg;
    if (!x || !q || !sfa || M <= 0 || K <= 0 || (x_dtype != DG_DTYPE_F32 && x_dtype != DG_DTYPE_BF16))
        return DG_ERR_INVALID_ARG;
    if (K % kQBlock != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sfa))
        return DG_ERR_MISALIGNED;
    DeviceInfo info;
    dg_status_t st = current_device(&info);
    if (st != DG_OK)
        return st;
    const int KB = K / kQBlock;
    // eight groups per warp keep eight 16-byte loads per lane in flight on
    // large problems (33152 x 7168 fp32: 191 against 213 us with four); a
    // problem with less than a full wave of such tasks takes four, and a small
    // one (less than a wave of four-group tasks) one group per warp, spreading
    // the division chains over more warps
    const long long rows8 = ceil_div(M, kQuantWarps);
    const long long wave = info.sm_count * 8LL;
    const int gpw = rows8 * ceil_div(KB, 8) >= wave ? 8 : rows8 * ceil_div(KB, 4) >= wave ? 4 : 1;
    const long long tasks = rows8 * ceil_div(KB, gpw);
    const int grid = static_cast<int>(tasks < wave ? tasks : wave);
    const int ldsfa = round_up(M, 4);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto run = [&](auto kernel, const auto *xt) {
        kernel<<<grid, kQuantWarps * 32, 0, s>>>(xt, q, sfa, M, K, ldsfa);
    };
    if (x_dtype == DG_DTYPE_F32) {
        const float *xf = static_cast<const float *>(x);
        if (gpw == 8)
            run(quant_act_1x128_kernel<float, 8>, xf);
        else if (gpw == 4)
            run(quant_act_1x128_kernel<float, 4>, xf);
        else
            run(quant_act_1x128_kernel<float, 1>, xf);
    } else {
        const uint16_t *xh = static_cast<const uint16_t *>(x);
        if (gpw == 8)
            run(quant_act_1x128_kernel<uint16_t, 8>, xh);
        else if (gpw == 4)
            run(quant_act_1x128_kernel<uint16_t, 4>, xh);
        else
            run(quant_act_1x128_kernel<uint16_t, 1>, xh);
    }
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

extern "C" dg_status_t dg_quant_weight_128x128(const float *w, uint8_t *q, float *sfb, int G, int N, int K,
                                               void *stream)
{
    using namespace dg;
    if (!w || !q || !sfb || G <= 0 || N <= 0 || K <= 0)
        return DG_ERR_INVALID_ARG;
    if (K % kQBlock != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(w) || !aligned16(q) || !aligned16(sfb))
        return DG_ERR_MISALIGNED;
    DeviceInfo info;
    dg_status_t st = current_device(&info);
    if (st != DG_OK)
        return st;
    const long long blocks = static_cast<long long>(G) * ceil_div(N, kQBlock) * (K / kQBlock);
    if (blocks > 0x7FFFFFFFLL)
        return DG_ERR_UNSUPPORTED_SHAPE;
    quant_weight_128x128_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        w, q, sfb, N, K);
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

extern "C" dg_status_t dg_quant_mx_1x32(const float *x, uint8_t *q, uint8_t *sx, int R, int K, void *stream)
{
    using namespace dg;
    if (!x || !q || !sx || R <= 0 || K <= 0)
        return DG_ERR_INVALID_ARG;
    if (K % 128 != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sx))
        return DG_ERR_MISALIGNED;
    DeviceInfo info;
    dg_status_t st = current_device(&info);
    if (st != DG_OK)
        return st;
    const long long tasks = static_cast<long long>(R) * (K / 128);
    const long long blocks = (tasks + 7) / 8;
    const int grid = static_cast<int>(blocks < info.sm_count * 16LL ? blocks : info.sm_count * 16LL);
    quant_mx_1x32_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, q, sx, R, K);
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}
