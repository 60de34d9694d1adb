// GEMMs whose accumulator stays in tensor memory across all of K, for the two
// formats the pages name beside per-group-scaled FP8 (2kiu.com DeepGEMM
// tutorial, 1 and 2.2: BF16; 7: MX / micro-scaling formats with finer scale
// granularity):
//
//   BF16   D = bf16_rn(sum_k A[m,k] B[n,k]) with bf16 operands
//          (tcgen05.mma kind::f16, fp32 accumulator);
//   MX     D = bf16_rn(sum_kb 2^(ea[m,kb] + eb[n,kb]) sum_{k in kb} A[m,k] B[n,k])
//          with E4M3 operands and one UE8M0 scale per 32 consecutive K values
//          of each row (OCP Microscaling v1.0), applied by the tensor core
//          (tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X): the
//          hardware scales every 32-wide block, so there is no promotion.
//
// Two kernels per format.  acc_pair_kernel (further down) computes 256 x 256
// tiles on pairs of SMs and takes every problem with at least half the SMs'
// worth of such tiles; acc_gemm_kernel, here, computes 128 x 256 tiles on one
// SM and takes the smaller ones.
//
// acc_gemm_kernel: one CTA per SM, persistent, 128 x 256 tiles.  A K block of
// such a tile brings 48 KB per 512 MMA cycles (one SM takes in at most ~80
// bytes per cycle through TMA), against 32 KB per 256 cycles for a 128 x 128
// tile.  Roles:
//   warp 0      TMA producer of A (one box of 128 rows x two 128-byte K
//               chunks per stage; it also arms the stage's full barrier);
//   warp 1      TMA producer of B (256 rows x two chunks);
//   warp 2      allocates TMEM; lane 0 issues the MMAs of every stage into
//               the tile's accumulator, commits each stage to its "empty"
//               barrier and the tile's last stage to the accumulator's "full"
//               barrier.  BF16: one MMA of N = 256 per K step, two
//               accumulators alternating by tile.  MX: two MMAs of N = 128 per
//               K step (B rows 0-127 and 128-255, each with its own scale
//               granule) into one accumulator: the scale columns take the
//               room of the second;
//   warps 4-7   (MX) scale writers: per stage and 128-wide K chunk, the
//               scales of the tile's 128 rows of A and of each 128-row half
//               of B (one 32-bit word per row: the scales of the chunk's four
//               32-wide blocks) go into one 4-column TMEM granule each with
//               tcgen05.st; the MMA of K step j selects byte j (the
//               instruction's scale-factor ID).  They arrive on the stage's
//               full barrier, so the issuer waits once per stage;
//   epilogue    (BF16: 4 warps of 256 columns; MX: 8 warps of 128) per tile,
//               once the accumulator is complete, each thread loads its row 32
//               columns at a time, rounds to bf16 and stores through shared
//               memory; the accumulator is released as soon as its TMEM loads
//               are done.
// Every wait is bounded (dg_wait.cuh).
#include <stdlib.h>

#include <algorithm>

#include "dg_common.h"
#include "dg_ptx.cuh"
#include "dg_wait.cuh"

namespace dg {
namespace {

// D[tmem] (+)= A . B^T for a CTA pair (M = 256): bf16 operands (kind::f16),
// each CTA holding its 128 rows of A and its half of B's rows at the same
// shared-memory offsets; D has this CTA's 128 rows in each CTA's TMEM.
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled MX MMA for a CTA pair (M = 256, N = 256): E4M3 operands with
// one UE8M0 scale per 32 K values.  At the same columns of each CTA's tensor
// memory: the granule of that CTA's own 128 rows of A at sfa_tmem, and the
// granules of all 256 rows of B at sfb_tmem (rows 0-127 in its first four
// columns, 128-255 in the next four), found by bit-exact tests: a granule of
// only the CTA's own half of B gave wrong columns 128-255.
__device__ __forceinline__ void mma_mx_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

constexpr int kAccKind_BF16 = 0;
constexpr int kAccKind_MX = 1;

constexpr int kABM = 128;
constexpr int kAKps = 2;                   // 128-byte K chunks per stage
constexpr int kAGroupM = 16;               // m-blocks per rasterisation band

template <int KIND>
struct AccCfg {
    static constexpr int kBN = 256;
    static constexpr int kStages = 2;
    static constexpr int kElemsPerChunk = KIND == kAccKind_BF16 ? 64 : 128;   // K values per 128-byte row
    static constexpr int kSfWarps = KIND == kAccKind_MX ? 4 : 0;
    static constexpr int kEpiWarp0 = 4 + kSfWarps;
    static constexpr int kEpiWarps = KIND == kAccKind_MX ? 8 : 4;
    static constexpr int kEpiCols = kBN / (kEpiWarps / 4);     // columns per epilogue warp
    static constexpr int kAccBufs = KIND == kAccKind_MX ? 1 : 2;
    static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
    static constexpr int kABox = kABM * 128 * kAKps;          // 32 KiB
    static constexpr int kBBox = kBN * 128 * kAKps;           // 64 KiB
    static constexpr int kAOff = 0;
    static constexpr int kBOff = kAOff + kStages * kABox;
    static constexpr int kOutRow = 32 * 2 + 16;               // 32 bf16 columns + 16 bytes of padding
    static constexpr int kOutOff = kBOff + kStages * kBBox;
    static constexpr int kBarOff = kOutOff + kEpiWarps * 32 * kOutRow;
    // full[S], empty[S], acc_full[2], acc_empty[2], drain
    static constexpr int kMiscOff = kBarOff + 8 * (2 * kStages + 5);
    static constexpr int kAlloc = kMiscOff + 16 + 1024;
    // TMEM: the accumulators (kBN columns each), then (MX) the scale columns
    // of every stage: per chunk one granule for A's scales and one for each
    // 128-row half of B's, each on its own 4-column (128-bit) boundary, the
    // granule in which scale factors are laid out in tensor memory
    static constexpr uint32_t kSfCol0 = kAccBufs * kBN;
    static constexpr uint32_t kSfStride = 12;                 // columns per chunk: A at +0, B halves at +4, +8
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSfCol0 % 4 == 0 && kSfStride % 4 == 0, "scale columns on 4-column boundaries");
    static_assert(kAccBufs * kBN + (KIND == kAccKind_MX ? kSfStride * kAKps * kStages : 0) <= 512, "TMEM columns");
    static_assert(kEpiWarps % 4 == 0 && kEpiCols % 32 == 0, "epilogue split");
    static_assert(kAlloc <= 232448, "shared memory");
};

// Instruction descriptors (fp32 accumulator, both operands K-major):
// kind::f16 with bf16 A and B (format 1 in bits 7-9 and 10-12), D format
// f32 (1) in bits 4-5; kind::mxf8f6f4 with E4M3 A and B (format 0), UE8M0
// scales (bit 23), the B and A scale-factor IDs (the byte of the scale word
// that this K step uses) in bits 4-5 and 29-30.  N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t idesc_mx_e4m3(uint32_t M, uint32_t N, uint32_t sf_id)
{
    return (sf_id << 4) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) | (sf_id << 29);
}

struct AccProblem {
    int M;
    int N;
    int K;
};

template <int KIND>
__global__ void __launch_bounds__(AccCfg<KIND>::kThreads, 1)
    acc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const uint8_t *__restrict__ sfa, const uint8_t *__restrict__ sfb, uint16_t *__restrict__ d,
                    AccProblem p, unsigned int *status)
{
    using C = AccCfg<KIND>;
    constexpr int BN = C::kBN;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    constexpr uint32_t kAB = C::kAccBufs;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::kMiscOff + 4);

    const int pM = p.M, pN = p.N, pK = p.K;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int KC = pK / C::kElemsPerChunk;        // 128-byte K chunks
    const int nst = (KC + kAKps - 1) / kAKps;     // stages per tile
    const int m_blocks = (pM + kABM - 1) / kABM;
    const int n_blocks = (pN + BN - 1) / BN;
    const int num_tiles = m_blocks * n_blocks;
    auto tile_mn = [m_blocks, n_blocks](int t, int &m0, int &n0) {
        const int band_tiles = kAGroupM * n_blocks;
        const int band = t / band_tiles;
        const int first = band * kAGroupM;
        const int band_m = min(m_blocks - first, kAGroupM);
        const int local = t - band * band_tiles;
        m0 = (first + local % band_m) * kABM;
        n0 = (local / band_m) * BN;
    };

    // ------------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // the A producer's arrive (with the stage's bytes) and, for MX,
            // one arrive per scale-writer warp
            mbar_init(full_bar(s), 1 + C::kSfWarps);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), C::kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    griddep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 2) {
        // ------------------------------------------------------- TMA producers
        if (lane == 0) {
            const bool is_a = warp == 0;
            const CUtensorMap *map = is_a ? &tmap_a : &tmap_b;
            const uint32_t dst0 = sbase + (is_a ? C::kAOff : C::kBOff);
            const uint32_t box = is_a ? C::kABox : C::kBBox;
            uint32_t gs = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                int m0, n0;
                tile_mn(t, m0, n0);
                for (int j = 0; j < nst; ++j, ++gs) {
                    const int s = static_cast<int>(gs % S);
                    if (!wait_phase(empty_bar(s), ((gs / S) & 1u) ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    if (is_a)
                        mbar_arrive_expect_tx(full_bar(s), C::kABox + C::kBBox);
                    tma_load_3d(dst0 + s * box, map, full_bar(s), 0, is_a ? m0 : n0, j * kAKps);
                }
            }
            if (!ok) {
                // copies in flight complete on full barriers this thread may
                // not observe; give them time to land before the CTA exits
                const long long t0 = clock64();
                while (clock64() - t0 < 20000000ll) {
                }
            }
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint64_t desc_a0 = smem_desc_sw128(sbase + C::kAOff);
            const uint64_t desc_b0 = smem_desc_sw128(sbase + C::kBOff);
            uint32_t gs = 0;
            uint32_t tcount = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++tcount) {
                const uint32_t buf = tcount % kAB;
                // the epilogue has released this accumulator's previous tile
                if (!wait_phase(acce_bar(buf), ((tcount / kAB) & 1u) ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int j = 0; j < nst; ++j, ++gs) {
                    const int s = static_cast<int>(gs % S);
                    const uint32_t ph = (gs / S) & 1u;
                    if (!wait_phase(full_bar(s), ph, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kAKps; ++c) {
                        const uint64_t da = desc_a0 + static_cast<uint64_t>((s * C::kABox + c * kABM * 128) >> 4);
                        const uint64_t db = desc_b0 + static_cast<uint64_t>((s * C::kBBox + c * BN * 128) >> 4);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            // K step k of chunk c: 32 bytes further along the row;
                            // the tile's first step overwrites the accumulator
                            const uint32_t acc = (j > 0 || c > 0 || k > 0) ? 1u : 0u;
                            if constexpr (KIND == kAccKind_BF16) {
                                mma_f16(d_tmem, da + 2 * k, db + 2 * k, idesc_bf16_f32(kABM, BN), acc);
                            } else {
                                // two MMAs of N = 128: B rows 0-127 into columns
                                // 0-127, rows 128-255 into 128-255
                                const uint32_t sf_col = tmem_base + C::kSfCol0 + C::kSfStride * (s * kAKps + c);
                                constexpr uint64_t kHalfB = (128 * 128) >> 4;
                                mma_mx(d_tmem, da + 2 * k, db + 2 * k, idesc_mx_e4m3(kABM, 128, k), sf_col, sf_col + 4,
                                       acc);
                                mma_mx(d_tmem + 128, da + 2 * k, db + kHalfB + 2 * k, idesc_mx_e4m3(kABM, 128, k), sf_col,
                                       sf_col + 8, acc);
                            }
                        }
                    }
                    mma_commit(empty_bar(s));
                }
                if (!ok)
                    break;
                mma_commit(accf_bar(buf));
            }
            // every MMA this thread issued has completed once this barrier flips
            mma_commit(drain_bar);
            drain_wait(drain_bar, 0);
        }
    } else if (KIND == kAccKind_MX && warp >= 4 && warp < C::kEpiWarp0) {
        // ------------------------------------------------------- scale writers
        // Tensor-memory layout of one 128-wide K chunk's scales for 128 rows
        // (one scale per 32 K values): a 4-column (128-bit) granule in which
        // lane l holds rows l, l + 32, l + 64 and l + 96 in columns 0-3, each
        // 32-bit cell carrying the four scales of that row's four 32-wide
        // blocks (byte j for K step j, the MMA's scale-factor ID), and every
        // 32-lane quarter holds the same copy.  So each of the four warps
        // writes the whole granules into its own quarter: thread l loads the
        // words of rows l + 32 i (A: 4 rows; B: 8, two granules).  A stage's
        // granules are rewritten only after its MMAs have completed (its
        // empty barrier).
        const int q = warp & 3;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + C::kSfCol0;
        // The stages of all this CTA's tiles in order; the words of the next
        // stage are loaded while the current one is written, into the other
        // of two fixed register sets (the loop is unrolled by two, so no
        // value moves between registers while its load is in flight).
        const int total = ((num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                           static_cast<int>(gridDim.x)) * nst;
        auto load_words = [&](int u, uint32_t (&w)[kAKps][12]) {
            if (u >= total) {
                return;
            }
            int m0, n0;
            tile_mn(static_cast<int>(blockIdx.x) + (u / nst) * static_cast<int>(gridDim.x), m0, n0);
            const int j = u % nst;
#pragma unroll
            for (int c = 0; c < kAKps; ++c) {
                const int kc = j * kAKps + c;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ma = m0 + lane + 32 * i;
                    w[c][i] = (ma < pM && kc < KC)
                                  ? __ldg(reinterpret_cast<const uint32_t *>(sfa) + static_cast<size_t>(kc) * pM + ma)
                                  : 0u;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int nb = n0 + lane + 32 * i;
                    w[c][4 + i] = (nb < pN && kc < KC)
                                      ? __ldg(reinterpret_cast<const uint32_t *>(sfb) + static_cast<size_t>(kc) * pN + nb)
                                      : 0u;
                }
            }
        };
        auto write_stage = [&](int u, uint32_t (&w)[kAKps][12]) -> bool {
            const uint32_t gs = static_cast<uint32_t>(u);
            const int s = static_cast<int>(gs % S);
            if (!__all_sync(0xffffffffu, wait_phase(empty_bar(s), ((gs / S) & 1u) ^ 1u, abort_flag, status)))
                return false;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kAKps; ++c) {
                const uint32_t col = t_lane + C::kSfStride * (s * kAKps + c);
                tmem_st4(col, w[c][0], w[c][1], w[c][2], w[c][3]);
                tmem_st4(col + 4, w[c][4], w[c][5], w[c][6], w[c][7]);
                tmem_st4(col + 8, w[c][8], w[c][9], w[c][10], w[c][11]);
            }
            tmem_wait_st();
            tc_fence_before();
            if (lane == 0)
                mbar_arrive(full_bar(s));
            return true;
        };
        uint32_t w0[kAKps][12], w1[kAKps][12];
        load_words(0, w0);
        for (int u = 0; u < total; u += 2) {
            load_words(u + 1, w1);
            if (!write_stage(u, w0))
                break;
            if (u + 1 >= total)
                break;
            load_words(u + 2, w0);
            if (!write_stage(u + 1, w1))
                break;
        }
    } else if (warp >= C::kEpiWarp0) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int e = warp - C::kEpiWarp0;
        const int col0 = (e >> 2) * C::kEpiCols;                 // this warp's columns of the tile
        const uint32_t stage_u32 = sbase + C::kOutOff + e * 32 * C::kOutRow;
        uint32_t tcount = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++tcount) {
            int m0, n0;
            tile_mn(t, m0, n0);
            const uint32_t buf = tcount % kAB;
            if (!__all_sync(0xffffffffu, wait_phase(accf_bar(buf), (tcount / kAB) & 1u, abort_flag, status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + col0;
            const int rows_left = pM - (m0 + q * 32);
            uint16_t *const d_warp = d + static_cast<size_t>(m0 + q * 32) * pN + n0 + col0;
#pragma unroll 1
            for (int c = 0; c < C::kEpiCols / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(t_acc + c * 32, v);
                tmem_wait_ld32(v);
                if (c == C::kEpiCols / 32 - 1) {
                    // the accumulator is free for the tile after next
                    tc_fence_before();
                    if (lane == 0)
                        mbar_arrive(acce_bar(buf));
                }
                // this thread's row: 32 bf16 values = 64 bytes, staged so that
                // the warp stores 8 rows x 64 bytes per instruction
                const uint32_t my_row = stage_u32 + lane * C::kOutRow;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    st_shared_v4(my_row + 16 * k, pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                                 pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                                 pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                                 pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
                __syncwarp();
                const int cols_left = pN - (n0 + col0 + c * 32);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int rr = h * 8 + (lane >> 2);
                    const int cc = lane & 3;
                    if (rr < rows_left && cc * 8 < cols_left) {
                        const uint4 w = ld_shared_v4(stage_u32 + rr * C::kOutRow + 16 * cc);
                        st_global_v4(d_warp + static_cast<size_t>(rr) * pN + c * 32 + cc * 8, w.x, w.y, w.z, w.w);
                    }
                }
                __syncwarp();
            }
        }
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// BF16 and MX on a CTA pair: 256 x 256 tiles computed by a cluster of two CTAs
// that share one tcgen05.mma of M = 256 (cta_group::2).  Each CTA holds its
// own 128 rows of A and half of the tile's 256 B rows, so a K chunk brings
// 32 KB per SM per 512 MMA cycles (63 bytes per cycle), within what one SM
// takes in through TMA (~80), where the one-SM 128 x 256 tile needs 94.
// Roles, in each CTA:
//   warp 0      TMA producer of A (this CTA's 128 rows, two chunks per box);
//   warp 1      TMA producer of B (this CTA's 128 of the tile's 256 rows); all
//               four copies of a stage complete on rank 0's full barrier,
//               armed by rank 0's warp 0;
//   warp 2      allocates the TMEM of both CTAs; on rank 0, lane 0 issues every
//               MMA and commits to both CTAs' barriers.  BF16: two
//               accumulators alternating by tile.  MX: one accumulator (the
//               scale columns take the room of the second);
//   warps 4-7   (MX) scale writers: per stage and 128-wide K chunk, the
//               granule of this CTA's 128 rows of A and the two granules of
//               the tile's 256 rows of B (the one-SM kernel's granule layout);
//               they arrive on rank 0's full barrier of the stage;
//   last 8      epilogue: 2 warps per TMEM lane quarter, 128 columns each;
//               they release the accumulator on rank 0's barrier as soon as
//               their TMEM loads are done, then store bf16.
// Every wait is bounded (dg_wait.cuh).
constexpr int kQRows = 128;                // rows per CTA
constexpr int kQBN = 256;                  // columns per pair tile
constexpr int kQStages = 3;
constexpr int kQEpiWarps = 8;
constexpr int kQEpiCols = kQBN / (kQEpiWarps / 4);
constexpr int kQGroupM = 8;                // pair rows per rasterisation band

template <int KIND>
struct PairAccCfg {
    static constexpr int kSfWarps = KIND == kAccKind_MX ? 4 : 0;
    static constexpr int kEpiWarp0 = 4 + kSfWarps;
    static constexpr int kThreads = 32 * (kEpiWarp0 + kQEpiWarps);
    static constexpr int kAccBufs = KIND == kAccKind_MX ? 1 : 2;
    static constexpr int kElemsPerChunk = KIND == kAccKind_BF16 ? 64 : 128;   // K values per 128-byte row
    static constexpr int kBox = kQRows * 128 * kAKps;         // 32 KiB
    static constexpr int kAOff = 0;
    static constexpr int kBOff = kAOff + kQStages * kBox;
    static constexpr int kOutRow = 32 * 2 + 16;               // 32 bf16 columns + 16 bytes of padding
    static constexpr int kOutOff = kBOff + kQStages * kBox;
    static constexpr int kBarOff = kOutOff + kQEpiWarps * 32 * kOutRow;
    // full[S], empty[S], acc_full[2], acc_empty[2], drain
    static constexpr int kMiscOff = kBarOff + 8 * (2 * kQStages + 5);
    static constexpr int kAlloc = kMiscOff + 16 + 1024;
    // TMEM: the accumulators, then (MX) per stage and chunk one granule for
    // A's scales and one for B's, each on its own 4-column boundary
    static constexpr uint32_t kSfCol0 = kAccBufs * kQBN;
    static constexpr uint32_t kSfStride = 12;                 // columns per chunk: A at +0, B rows 0-127 at +4, 128-255 at +8
    static_assert(kAlloc <= 232448, "shared memory per CTA");
    static_assert(kSfCol0 % 4 == 0 && kSfStride % 4 == 0, "scale columns on 4-column boundaries");
    static_assert(kAccBufs * kQBN + (KIND == kAccKind_MX ? kSfStride * kAKps * kQStages : 0) <= 512, "TMEM columns");
};

template <int KIND>
__global__ void __launch_bounds__(PairAccCfg<KIND>::kThreads, 1)
    acc_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const uint8_t *__restrict__ sfa, const uint8_t *__restrict__ sfb, uint16_t *__restrict__ d,
                    AccProblem p, unsigned int *status)
{
    using L = PairAccCfg<KIND>;
    constexpr int S = kQStages;
    constexpr uint32_t kAB = L::kAccBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::kMiscOff + 4);

    const int pM = p.M, pN = p.N, pK = p.K;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair_id = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int KC = pK / L::kElemsPerChunk;         // 128-byte K chunks
    const int nst = (KC + kAKps - 1) / kAKps;      // stages per tile
    const int m_blocks = (pM + 2 * kQRows - 1) / (2 * kQRows);
    const int n_blocks = (pN + kQBN - 1) / kQBN;
    const int num_tiles = m_blocks * n_blocks;
    auto tile_mn = [m_blocks, n_blocks](int t, int &m0, int &n0) {
        const int band_tiles = kQGroupM * n_blocks;
        const int band = t / band_tiles;
        const int first = band * kQGroupM;
        const int band_m = min(m_blocks - first, kQGroupM);
        const int local = t - band * band_tiles;
        m0 = (first + local % band_m) * 2 * kQRows;
        n0 = (local / band_m) * kQBN;
    };

    // ------------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // rank 0's producer arms it (and, for MX, the scale writers of
            // both CTAs arrive); all four copies complete it
            mbar_init(full_bar(s), 1 + 2 * L::kSfWarps);
            mbar_init(empty_bar(s), 1);         // the issuer's commit, multicast to both CTAs
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * kQEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    griddep_wait();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    // rank 0's copies of the shared barriers, as shared::cluster addresses
    const uint32_t full0 = mapa_shared(full_bar(0), 0);
    const uint32_t acce0 = mapa_shared(acce_bar(0), 0);

    if (warp < 2) {
        // ------------------------------------------------------- TMA producers
        if (lane == 0) {
            const bool is_a = warp == 0;
            const CUtensorMap *map = is_a ? &tmap_a : &tmap_b;
            const uint32_t dst0 = sbase + (is_a ? L::kAOff : L::kBOff);
            uint32_t gs = 0;
            bool ok = true;
            for (int t = pair_id; ok && t < num_tiles; t += num_pairs) {
                int m0, n0;
                tile_mn(t, m0, n0);
                const int row = (is_a ? m0 : n0) + static_cast<int>(rank) * kQRows;
                for (int j = 0; j < nst; ++j, ++gs) {
                    const int s = static_cast<int>(gs % S);
                    if (!wait_phase(empty_bar(s), ((gs / S) & 1u) ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    if (is_a && rank == 0)
                        mbar_arrive_expect_tx(full_bar(s), 4u * L::kBox);
                    tma_load_3d_pair(dst0 + s * L::kBox, map, full0 + 8u * s, 0, row, j * kAKps);
                }
            }
            if (!ok) {
                // copies in flight complete on rank 0's full barriers, which
                // this thread may not observe: give them time to land
                const long long t0 = clock64();
                while (clock64() - t0 < 20000000ll) {
                }
            }
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------- MMA issuer
        if (rank == 0 && lane == 0) {
            const uint64_t desc_a0 = smem_desc_sw128(sbase + L::kAOff);
            const uint64_t desc_b0 = smem_desc_sw128(sbase + L::kBOff);
            uint32_t gs = 0;
            uint32_t tcount = 0;
            bool ok = true;
            for (int t = pair_id; ok && t < num_tiles; t += num_pairs, ++tcount) {
                const uint32_t buf = tcount % kAB;
                // the epilogues of both CTAs have released this accumulator
                if (!wait_phase(acce_bar(buf), ((tcount / kAB) & 1u) ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * kQBN;
                for (int j = 0; j < nst; ++j, ++gs) {
                    const int s = static_cast<int>(gs % S);
                    if (!wait_phase(full_bar(s), (gs / S) & 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kAKps; ++c) {
                        const uint32_t off = static_cast<uint32_t>(s * L::kBox + c * kQRows * 128) >> 4;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t acc = (j > 0 || c > 0 || k > 0) ? 1u : 0u;
                            if constexpr (KIND == kAccKind_BF16) {
                                mma_f16_pair(d_tmem, desc_a0 + off + 2 * k, desc_b0 + off + 2 * k,
                                             idesc_bf16_f32(2 * kQRows, kQBN), acc);
                            } else {
                                const uint32_t sf_col = tmem_base + L::kSfCol0 + L::kSfStride * (s * kAKps + c);
                                mma_mx_pair(d_tmem, desc_a0 + off + 2 * k, desc_b0 + off + 2 * k,
                                            idesc_mx_e4m3(2 * kQRows, kQBN, k), sf_col, sf_col + 4, acc);
                            }
                        }
                    }
                    mma_commit_pair_mc(empty_bar(s), 3);
                }
                if (!ok)
                    break;
                mma_commit_pair_mc(accf_bar(buf), 3);
            }
            // every MMA this thread issued has completed once this barrier flips
            mma_commit_pair_mc(drain_bar, 1);
            drain_wait(drain_bar, 0);
        }
    } else if (KIND == kAccKind_MX && warp >= 4 && warp < L::kEpiWarp0) {
        // ------------------------------------------------------- scale writers
        // Granule layout as in the one-SM kernel (lane l holds rows l, l + 32,
        // l + 64, l + 96 of a 128-row block in columns 0-3, byte j = K step j,
        // the same copy in every 32-lane quarter), for this CTA's 128 rows of
        // A and for both 128-row halves of the tile's B.  The words of the
        // next stage are loaded while the current one is written, into the
        // other of two fixed register sets.
        const int q = warp & 3;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + L::kSfCol0;
        const int total = ((num_tiles - pair_id + num_pairs - 1) / num_pairs) * nst;
        auto load_words = [&](int u, uint32_t (&w)[kAKps][12]) {
            if (u >= total)
                return;
            int m0, n0;
            tile_mn(pair_id + (u / nst) * num_pairs, m0, n0);
            const int j = u % nst;
            const int ma0 = m0 + static_cast<int>(rank) * kQRows + lane;
            const int nb0 = n0 + lane;
#pragma unroll
            for (int c = 0; c < kAKps; ++c) {
                const int kc = j * kAKps + c;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ma = ma0 + 32 * i;
                    w[c][i] = (ma < pM && kc < KC)
                                  ? __ldg(reinterpret_cast<const uint32_t *>(sfa) + static_cast<size_t>(kc) * pM + ma)
                                  : 0u;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int nb = nb0 + 32 * i;
                    w[c][4 + i] = (nb < pN && kc < KC)
                                      ? __ldg(reinterpret_cast<const uint32_t *>(sfb) + static_cast<size_t>(kc) * pN + nb)
                                      : 0u;
                }
            }
        };
        auto write_stage = [&](int u, uint32_t (&w)[kAKps][12]) -> bool {
            const uint32_t gs = static_cast<uint32_t>(u);
            const int s = static_cast<int>(gs % S);
            if (!__all_sync(0xffffffffu, wait_phase(empty_bar(s), ((gs / S) & 1u) ^ 1u, abort_flag, status)))
                return false;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kAKps; ++c) {
                const uint32_t col = t_lane + L::kSfStride * (s * kAKps + c);
                tmem_st4(col, w[c][0], w[c][1], w[c][2], w[c][3]);
                tmem_st4(col + 4, w[c][4], w[c][5], w[c][6], w[c][7]);
                tmem_st4(col + 8, w[c][8], w[c][9], w[c][10], w[c][11]);
            }
            tmem_wait_st();
            tc_fence_before();
            if (lane == 0)
                mbar_arrive_cluster(full0 + 8u * s);
            return true;
        };
        uint32_t w0[kAKps][12], w1[kAKps][12];
        load_words(0, w0);
        for (int u = 0; u < total; u += 2) {
            load_words(u + 1, w1);
            if (!write_stage(u, w0))
                break;
            if (u + 1 >= total)
                break;
            load_words(u + 2, w0);
            if (!write_stage(u + 1, w1))
                break;
        }
    } else if (warp >= L::kEpiWarp0) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int e = warp - L::kEpiWarp0;
        const int col0 = (e >> 2) * kQEpiCols;
        const uint32_t stage_u32 = sbase + L::kOutOff + e * 32 * L::kOutRow;
        uint32_t tcount = 0;
        bool ok = true;
        for (int t = pair_id; ok && t < num_tiles; t += num_pairs, ++tcount) {
            int m0, n0;
            tile_mn(t, m0, n0);
            const uint32_t buf = tcount % kAB;
            if (!__all_sync(0xffffffffu, wait_phase(accf_bar(buf), (tcount / kAB) & 1u, abort_flag, status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kQBN + col0;
            const int row0 = m0 + static_cast<int>(rank) * kQRows + q * 32;   // this warp's first row
            const int rows_left = pM - row0;
            uint16_t *const d_warp = d + static_cast<size_t>(row0) * pN + n0 + col0;
#pragma unroll 1
            for (int c = 0; c < kQEpiCols / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(t_acc + c * 32, v);
                tmem_wait_ld32(v);
                if (c == kQEpiCols / 32 - 1) {
                    // the accumulator is free for its next tile
                    tc_fence_before();
                    if (lane == 0)
                        mbar_arrive_cluster(acce0 + 8u * buf);
                }
                // this thread's row: 32 bf16 values = 64 bytes, staged so that
                // the warp stores 8 rows x 64 bytes per instruction
                const uint32_t my_row = stage_u32 + lane * L::kOutRow;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    st_shared_v4(my_row + 16 * k, pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                                 pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                                 pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                                 pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
                __syncwarp();
                const int cols_left = pN - (n0 + col0 + c * 32);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int rr = h * 8 + (lane >> 2);
                    const int cc = lane & 3;
                    if (rr < rows_left && cc * 8 < cols_left) {
                        const uint4 w = ld_shared_v4(stage_u32 + rr * L::kOutRow + 16 * cc);
                        st_global_v4(d_warp + static_cast<size_t>(rr) * pN + c * 32 + cc * 8, w.x, w.y, w.z, w.w);
                    }
                }
                __syncwarp();
            }
        }
    }

    // ------------------------------------------------------------- teardown
    // neither CTA leaves while the other may still signal its barriers or
    // read its tensor memory
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

// Whether the pair kernel takes a BF16 or MX problem: enough 256 x 256 tiles
// for half the SMs' worth of pairs (otherwise the one-SM kernel's 128 x 256
// tiles spread the work over more SMs).  DG_FORCE_ACC_PAIR = 1 / 0 overrides.
bool acc_pair_ok(int M, int N, int num_sms)
{
    const char *f = getenv("DG_FORCE_ACC_PAIR");
    if (f && f[0] == '1')
        return num_sms >= 2;
    if (f && f[0] == '0')
        return false;
    const int tiles = ceil_div(M, 2 * kQRows) * ceil_div(N, kQBN);
    return num_sms >= 2 && tiles >= num_sms / 2;
}

template <int KIND>
dg_status_t launch_acc_pair(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb, uint16_t *d, int M,
                            int N, int K, void *stream, const DeviceInfo &info)
{
    using L = PairAccCfg<KIND>;
    // operands viewed as [K chunks][rows][128 bytes]; a box is 128 bytes x
    // 128 rows x two chunks, 128-byte swizzled
    const int esize = KIND == kAccKind_BF16 ? 2 : 1;
    const CUtensorMapDataType dt = KIND == kAccKind_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t inner = 128 / esize;
    const uint64_t KC = static_cast<uint64_t>(K) / inner;
    CUtensorMap ta, tb;
    dg_status_t st;
    {
        const uint64_t dims[3] = {inner, static_cast<uint64_t>(M), KC};
        const uint64_t strides[2] = {static_cast<uint64_t>(K) * esize, 128};
        const uint32_t box[3] = {static_cast<uint32_t>(inner), kQRows, kAKps};
        st = encode_tensor_map(&ta, dt, 3, a, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    {
        const uint64_t dims[3] = {inner, static_cast<uint64_t>(N), KC};
        const uint64_t strides[2] = {static_cast<uint64_t>(K) * esize, 128};
        const uint32_t box[3] = {static_cast<uint32_t>(inner), kQRows, kAKps};
        st = encode_tensor_map(&tb, dt, 3, b, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    st = ensure_smem_attr(reinterpret_cast<const void *>(acc_pair_kernel<KIND>), L::kAlloc);
    if (st != DG_OK)
        return st;
    const int tiles = ceil_div(M, 2 * kQRows) * ceil_div(N, kQBN);
    const int pairs = std::min(info.sm_count / 2, std::max(1, tiles));
    AccProblem prob{M, N, K};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, acc_pair_kernel<KIND>, ta, tb, sfa, sfb, d, prob, info.status_word) != cudaSuccess)
        return DG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

template <int KIND>
dg_status_t launch_acc(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb, uint16_t *d, int M, int N,
                       int K, void *stream)
{
    using C = AccCfg<KIND>;
    DeviceInfo info;
    dg_status_t st = current_device(&info);
    if (st != DG_OK)
        return st;
    // operands viewed as [rows][K chunks][128 bytes]; a box is 128 bytes x
    // rows x two chunks, 128-byte swizzled (the FP8 GEMM's layout)
    const int esize = KIND == kAccKind_BF16 ? 2 : 1;
    const CUtensorMapDataType dt = KIND == kAccKind_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t inner = 128 / esize;
    const uint64_t KC = static_cast<uint64_t>(K) / inner;
    CUtensorMap ta, tb;
    {
        const uint64_t dims[3] = {inner, static_cast<uint64_t>(M), KC};
        const uint64_t strides[2] = {static_cast<uint64_t>(K) * esize, 128};
        const uint32_t box[3] = {static_cast<uint32_t>(inner), kABM, kAKps};
        st = encode_tensor_map(&ta, dt, 3, a, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    {
        const uint64_t dims[3] = {inner, static_cast<uint64_t>(N), KC};
        const uint64_t strides[2] = {static_cast<uint64_t>(K) * esize, 128};
        const uint32_t box[3] = {static_cast<uint32_t>(inner), static_cast<uint32_t>(C::kBN), kAKps};
        st = encode_tensor_map(&tb, dt, 3, b, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    st = ensure_smem_attr(reinterpret_cast<const void *>(acc_gemm_kernel<KIND>), C::kAlloc);
    if (st != DG_OK)
        return st;
    const int tiles = ceil_div(M, kABM) * ceil_div(N, C::kBN);
    AccProblem prob{M, N, K};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(tiles, info.sm_count));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kAlloc;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, acc_gemm_kernel<KIND>, ta, tb, sfa, sfb, d, prob, info.status_word) != cudaSuccess)
        return DG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

}  // namespace
}  // namespace dg

extern "C" dg_status_t dg_bf16_gemm_nt(const uint16_t *a, const uint16_t *b, uint16_t *d, int M, int N, int K,
                                       void *stream)
{
    if (!a || !b || !d || M <= 0 || N <= 0 || K <= 0)
        return DG_ERR_INVALID_ARG;
    if (K % 64 != 0 || N % 8 != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!dg::aligned16(a) || !dg::aligned16(b) || !dg::aligned16(d))
        return DG_ERR_MISALIGNED;
    dg::DeviceInfo info;
    const dg_status_t st = dg::current_device(&info);
    if (st != DG_OK)
        return st;
    if (dg::acc_pair_ok(M, N, info.sm_count))
        return dg::launch_acc_pair<dg::kAccKind_BF16>(a, nullptr, b, nullptr, d, M, N, K, stream, info);
    return dg::launch_acc<dg::kAccKind_BF16>(a, nullptr, b, nullptr, d, M, N, K, stream);
}

extern "C" dg_status_t dg_mx_gemm_nt(const uint8_t *a, const uint8_t *sa, const uint8_t *b, const uint8_t *sb,
                                     uint16_t *d, int M, int N, int K, void *stream)
{
    if (!a || !sa || !b || !sb || !d || M <= 0 || N <= 0 || K <= 0)
        return DG_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 8 != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!dg::aligned16(a) || !dg::aligned16(sa) || !dg::aligned16(b) || !dg::aligned16(sb) || !dg::aligned16(d))
        return DG_ERR_MISALIGNED;
    dg::DeviceInfo info;
    const dg_status_t st = dg::current_device(&info);
    if (st != DG_OK)
        return st;
    if (dg::acc_pair_ok(M, N, info.sm_count))
        return dg::launch_acc_pair<dg::kAccKind_MX>(a, sa, b, sb, d, M, N, K, stream, info);
    return dg::launch_acc<dg::kAccKind_MX>(a, sa, b, sb, d, M, N, K, stream);
}
