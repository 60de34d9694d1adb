// FP8 (E4M3) GEMM with fine-grained scaling and two-level accumulation on a
// pair of SMs: 256 x 256 tiles computed by a cluster of two CTAs sharing one
// tcgen05 MMA of M = 256 (cta_group::2), for the dense and MoE-contiguous
// layouts with bf16 output.
//
// What it computes is what fp8_gemm_kernel computes ("DeepGEMM：一款支持FP8通用
// 矩阵乘法(GEMM)的开源库", 技术细节/两级累加技术): per 128-wide K block kb the tensor
// cores form P_kb = A[:, kb] . B[:, kb]^T in fp32 and the CUDA cores promote it,
//     acc[m,n] = fmaf(P_kb[m,n], sfa[kb][m] * sfb[n/128][kb], acc[m,n]),
// kb ascending; D = bf16_rn(acc).  The results are the same bits.
//
// Why a pair.  On GB300 one SM takes in at most ~80 bytes per cycle from L2
// through TMA (with two or three issuing threads; one thread reaches 63-70),
// while the FP8 tensor core consumes a 128-row K block of A and of B per 2N
// cycles.  A 128 x 192 tile (one SM) needs 104 bytes per cycle; in a
// pair each SM holds its own 128 rows of A and half of B's 256 rows, so a
// K block brings 32 KB per SM per 512 MMA cycles (63 bytes per cycle), moved
// as 32 KB boxes (two K blocks per copy).
//
// Roles (the page's 线程专业化技术, redone for the pair), in each CTA:
//   warp 0      TMA producer of A: this CTA's 128 rows, two K blocks per box;
//   warp 1      TMA producer of B: this CTA's 128 of the tile's 256 B rows;
//               both copies of both CTAs complete on rank 0's "full"
//               barrier of the stage, armed by rank 0's warp 0;
//   warps 2, 3  (rank 0 only) MMA issuers: issuer i takes the i-th K block
//               of every stage into TMEM slot i (256 columns), 4 MMAs of
//               256 x 256 x 32, then commits to both CTAs' "tfull" barrier
//               of the slot and "empty" barrier of the stage; warp 2 also
//               allocates the TMEM columns (in both CTAs), warp 3 first builds
//               the contiguous layout's list of row pairs;
//   warps 4-19  epilogue: four warpgroups of 64 columns; a thread owns one
//               row (TMEM lane) of its CTA's 128.  Per K block it loads its
//               64 partial sums from TMEM, releases the slot (an arrive on
//               rank 0's "tempty" barrier, 32 arrivals from the two CTAs)
//               and FMAs them into fp32 registers with sfa * sfb; after the
//               last K block it stores bf16 through shared memory.
// The issuing threads never wait on a barrier while they could be issuing
// more work: a thread that polls an mbarrier stalls until its own earlier
// copies or MMAs have progressed, so the copies of A and B come from two
// threads and the K blocks alternate between two issuers.
//
// Waits are CTA-scope polls of the local barrier; arrivals from the peer CTA
// use the default (CTA-scope release) form: the work they order is complete
// (loads waited for, copies counted by the barrier's transaction bytes), and
// a cluster-scope release costs about a microsecond per handoff.
//
// Every wait is bounded (dg_wait.cuh); a timed-out role raises the CTA's
// abort flag and DG_DEVFLAG_TIMEOUT, and the CTA drains what it started
// before the pair meets at the final cluster barrier.
#include <stdlib.h>

#include "dg_common.h"
#include "dg_ptx.cuh"
#include "dg_wait.cuh"

namespace dg {
namespace {

constexpr int kPRowsCta = 128;             // rows per CTA (TMEM lanes)
constexpr int kPBN = 256;                  // columns per pair tile
constexpr int kPKps = 2;                   // K blocks per stage (one box per operand per CTA)
constexpr int kPStages = 2;
constexpr int kPEpiWarp0 = 4;
constexpr int kPEpiWarps = 16;             // 4 warpgroups x 64 columns
constexpr int kPEpiCols = 64;
constexpr int kPThreads = 32 * (kPEpiWarp0 + kPEpiWarps);
constexpr int kPGroupM = 8;                // pair rows per rasterisation band
constexpr uint32_t kPTmemCols = 512;       // two slots of 256 columns

struct PairSmem {
    static constexpr int kBox = kPRowsCta * 128 * kPKps;       // 32 KiB: 128 rows x 2 K blocks
    static constexpr int kAOff = 0;
    static constexpr int kBOff = kAOff + kPStages * kBox;
    // output staging: per epilogue warp its 32 rows x 64 bf16 columns (128
    // bytes a row), in the 128-byte swizzled order of the output's TMA store
    static constexpr int kOutWarpBytes = 32 * 128;
    static constexpr int kOutOff = kBOff + kPStages * kBox;
    // scales: per epilogue warp and stage parity, sfa of its 32 rows for the
    // stage's two K blocks and the two sfb values of its column block
    static constexpr int kScaleWarpBytes = 2 * (2 * 32 + 4) * 4;
    static constexpr int kScaleOff = kOutOff + kPEpiWarps * kOutWarpBytes;
    // re-quantised output: each row's amax over its 64 columns, per column
    // slice and tile parity, exchanged between the two slices of a
    // 128-column scale group
    static constexpr int kAmaxOff = kScaleOff + kPEpiWarps * kScaleWarpBytes;
    static constexpr int kBarOff = kAmaxOff + 2 * (kPBN / kPEpiCols) * kPRowsCta * 4;
    // full[S], empty[S], tfull[2], tempty[2], drain[2], xchg[4 quarters x 2 groups]
    static constexpr int kNumBars = 2 * kPStages + 6 + 8;
    static constexpr int kMiscOff = kBarOff + 256;             // tmem base, abort flag, pair-row count
    static constexpr int kListOff = kMiscOff + 16;
    static constexpr int kBytes = kListOff + kPairMaxRows * 4;
    static constexpr int kAlloc = kBytes + 1024;              // slack to align the base to 1024
    static_assert(kNumBars * 8 <= 256, "barrier area");
};

struct PairProblem {
    int M;        // dense: rows; contiguous: sum_M
    int N;
    int K;
    int G;
    int layout;
    int ldsfa;
};

struct PairTile {
    int m_cta;      // first row of A / D handled by this CTA (global row index)
    int rows;       // rows of this CTA's half that are stored (0..128)
    int n0;         // first column of the pair tile
    int g;          // expert (contiguous) or 0
};

// Tile t of the pair's sequence.  Dense: pair row p covers rows 256p..256p+255.
// Contiguous: pair row p is list[p], the first of one or two consecutive
// 128-row blocks of one expert; when it holds one block, rank 1 computes a
// copy of rank 0's block and stores nothing.
__device__ __forceinline__ PairTile pair_tile(int t, int rows_p, int n_blocks, int M, int layout, const int *list,
                                              const int32_t *meta, uint32_t rank)
{
    const int band_tiles = kPGroupM * n_blocks;
    const int band = t / band_tiles;
    const int first = band * kPGroupM;
    const int band_m = min(rows_p - first, kPGroupM);
    const int local = t - band * band_tiles;
    const int pr = first + local % band_m;
    PairTile ti;
    ti.n0 = (local / band_m) * kPBN;
    if (layout == DG_LAYOUT_DENSE) {
        ti.m_cta = pr * 2 * kPRowsCta + static_cast<int>(rank) * kPRowsCta;
        ti.rows = max(0, min(kPRowsCta, M - ti.m_cta));
        ti.g = 0;
    } else {
        const int e = list[pr];
        const int b0 = e & 0x7FFFFFFF;
        const bool two = (e >> 31) & 1;
        ti.m_cta = (b0 + ((two && rank) ? 1 : 0)) * kPRowsCta;
        ti.rows = (rank == 0 || two) ? kPRowsCta : 0;
        ti.g = meta[static_cast<size_t>(b0) * kPRowsCta];
    }
    return ti;
}

// QOUT: instead of bf16 D, write D re-quantised as the next GEMM's activation
// operand (E4M3 codes in D's layout and one fp32 scale per 1x128 group of each
// row, M-major), each group computed from the bf16-rounded values exactly as
// the 1x128 quantiser does; the same output as fp8_gemm_kernel's.
template <bool QOUT>
__global__ void __launch_bounds__(kPThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_d,
                         const float *__restrict__ sfa, const float *__restrict__ sfb, uint16_t *__restrict__ d,
                         uint8_t *__restrict__ qout, float *__restrict__ sfo,
                         const int32_t *__restrict__ meta, PairProblem p, unsigned int *status)
{
    using L = PairSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kPStages + s); };
    auto tfull_bar = [&](int i) { return bar0 + 8u * (2 * kPStages + i); };
    auto tempty_bar = [&](int i) { return bar0 + 8u * (2 * kPStages + 2 + i); };
    auto drain_bar = [&](int i) { return bar0 + 8u * (2 * kPStages + 4 + i); };
    // the two 64-column slices of 128-column scale group h in lane quarter q
    auto xchg_bar = [&](int q, int h) { return bar0 + 8u * (2 * kPStages + 6 + 2 * q + h); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::kMiscOff + 4);
    int *num_rows_s = reinterpret_cast<int *>(smem + L::kMiscOff + 8);
    int *list = reinterpret_cast<int *>(smem + L::kListOff);

    // the problem's fields as plain values (a reference to the parameter
    // would make the compiler copy it to local memory)
    const int pM = p.M, pN = p.N, pG = p.G, player = p.layout, pldsfa = p.ldsfa;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair_id = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int KB = p.K / 128;
    const int nst = (KB + kPKps - 1) / kPKps;   // stages per tile
    const int n_blocks = (pN + kPBN - 1) / kPBN;
    const int NBs = (pN + 127) / 128;

    // ------------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(full_bar(s), 1);      // rank 0's producer arms it; all four copies complete it
            mbar_init(empty_bar(s), 2);     // one commit from each issuer
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull_bar(i), 1);
            mbar_init(tempty_bar(i), 2 * kPEpiWarps);
            mbar_init(drain_bar(i), 1);
        }
        if constexpr (QOUT)
            for (int i = 0; i < 8; ++i)
                mbar_init(xchg_bar(i >> 1, i & 1), 64);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(tmem_slot), kPTmemCols);
        tmem_relinquish_pair();
    }
    griddep_wait();
    if (warp == 3) {
        int rows_p = 0;
        if (player == DG_LAYOUT_DENSE) {
            rows_p = (pM + 2 * kPRowsCta - 1) / (2 * kPRowsCta);
        } else {
            // Pair consecutive 128-row blocks of the same expert.  Block b's
            // expert is m_indices[128 b]; a block starts a pair at an even
            // position within its run of equal experts.
            const int nblk = pM / kPRowsCta;
            int carry_e = -2, carry_start = 0;
            for (int base = 0; base < nblk; base += 32) {
                const int b = base + lane;
                const int e = b < nblk ? meta[static_cast<size_t>(b) * kPRowsCta] : -3;
                int prev = __shfl_up_sync(0xffffffffu, e, 1);
                if (lane == 0)
                    prev = carry_e;
                const bool start = b < nblk && (b == 0 || e != prev);
                int rs = start ? b : -1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, rs, o);
                    if (lane >= o)
                        rs = max(rs, v);
                }
                rs = max(rs, carry_start);
                const bool valid = b < nblk && e >= 0 && e < pG;
                if (b < nblk && e >= pG)
                    raise_status(status, DG_DEVFLAG_BAD_EXPERT);
                const bool pstart = valid && ((b - rs) & 1) == 0;
                int nxt = __shfl_down_sync(0xffffffffu, e, 1);
                if (lane == 31)
                    nxt = (b + 1 < nblk) ? meta[static_cast<size_t>(b + 1) * kPRowsCta] : -3;
                const bool two = pstart && b + 1 < nblk && nxt == e;
                const uint32_t ball = __ballot_sync(0xffffffffu, pstart);
                if (pstart)
                    list[rows_p + __popc(ball & ((1u << lane) - 1u))] = b | (two ? static_cast<int>(0x80000000u) : 0);
                rows_p += __popc(ball);
                carry_e = __shfl_sync(0xffffffffu, e, 31);
                carry_start = __shfl_sync(0xffffffffu, rs, 31);
            }
        }
        if (lane == 0)
            *num_rows_s = rows_p;
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    const int rows_p = *num_rows_s;
    const int num_tiles = rows_p * n_blocks;
    const uint32_t tmem_base = *tmem_slot;
    // rank 0's copies of the shared barriers, as shared::cluster addresses
    const uint32_t full0 = mapa_shared(full_bar(0), 0);
    const uint32_t tempty0 = mapa_shared(tempty_bar(0), 0);

    if (warp < 2) {
        // ------------------------------------------------------- TMA producers
        if (lane == 0) {
            const bool is_a = warp == 0;
            const CUtensorMap *map = is_a ? &tmap_a : &tmap_b;
            const uint32_t dst0 = sbase + (is_a ? L::kAOff : L::kBOff);
            uint32_t gs = 0;
            bool ok = true;
            for (int t = pair_id; ok && t < num_tiles; t += num_pairs) {
                const PairTile ti = pair_tile(t, rows_p, n_blocks, pM, player, list, meta, rank);
                const int row = is_a ? ti.m_cta : ti.n0 + static_cast<int>(rank) * kPRowsCta;
                for (int j = 0; j < nst; ++j, ++gs) {
                    const int s = static_cast<int>(gs % kPStages);
                    const uint32_t ph = (gs / kPStages) & 1u;
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8u * s;
                    if (is_a && leader)
                        mbar_arrive_expect_tx(full_bar(s), 4u * L::kBox);
                    const uint32_t dst = dst0 + s * L::kBox;
                    if (is_a || player == DG_LAYOUT_DENSE)
                        tma_load_3d_pair(dst, map, fb, 0, row, j * kPKps);
                    else
                        tma_load_4d_pair(dst, map, fb, 0, row, j * kPKps, ti.g);
                }
            }
            if (!ok) {
                // The copies already issued complete on rank 0's full barriers,
                // which this thread may not be able to observe: give them time
                // to land (they take microseconds) before the CTA can exit.
                const long long t0 = clock64();
                while (clock64() - t0 < 20000000ll) {
                }
            }
        }
    } else if (warp < kPEpiWarp0) {
        // ------------------------------------------------------- MMA issuers
        if (leader && lane == 0) {
            const uint32_t me = static_cast<uint32_t>(warp - 2);
            constexpr uint32_t kIdesc = idesc_e4m3_f32(2 * kPRowsCta, kPBN);
            const uint64_t desc_a0 = smem_desc_sw128(sbase + L::kAOff);
            const uint64_t desc_b0 = smem_desc_sw128(sbase + L::kBOff);
            const uint32_t d_tmem = tmem_base + me * kPBN;
            uint32_t gs = 0;
            bool ok = true;
            for (int t = pair_id; ok && t < num_tiles; t += num_pairs) {
                for (int j = 0; j < nst; ++j, ++gs) {
                    const int s = static_cast<int>(gs % kPStages);
                    const uint32_t ph = (gs / kPStages) & 1u;
                    // the data first (its copies have normally landed long
                    // before), then the slot.  This thread takes one K block
                    // of every stage, so it has seen every earlier phase of
                    // the stage's full barrier: the barrier is never two
                    // phases behind when it is tested.
                    if (!wait_phase(full_bar(s), ph, abort_flag, status) ||
                        !wait_phase(tempty_bar(me), (gs & 1u) ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t off = static_cast<uint32_t>(s * L::kBox + me * (L::kBox / kPKps)) >> 4;
                    const uint64_t da = desc_a0 + off;
                    const uint64_t db = desc_b0 + off;
                    mma_f8f6f4_pair<false>(d_tmem, da, db, kIdesc);
                    mma_f8f6f4_pair<true>(d_tmem, da + 2, db + 2, kIdesc);
                    mma_f8f6f4_pair<true>(d_tmem, da + 4, db + 4, kIdesc);
                    mma_f8f6f4_pair<true>(d_tmem, da + 6, db + 6, kIdesc);
                    mma_commit_pair_mc(tfull_bar(me), 3);
                    mma_commit_pair_mc(empty_bar(s), 3);
                }
            }
            // every MMA this thread issued has completed once this barrier flips
            mma_commit_pair_mc(drain_bar(me), 1);
            drain_wait(drain_bar(me), 0);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                                   // TMEM lane quarter
        const int grp = (warp - kPEpiWarp0) >> 2;                 // 64-column slice
        const int r = q * 32 + lane;                              // row within this CTA's 128
        const int c0 = grp * kPEpiCols;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c0;
        const uint32_t stage_u32 = sbase + L::kOutOff + (warp - kPEpiWarp0) * L::kOutWarpBytes;
        const uint32_t scale_u32 = sbase + L::kScaleOff + (warp - kPEpiWarp0) * L::kScaleWarpBytes;
        uint32_t gs = 0;
        uint32_t tile_par = 0;   // alternates per tile (the re-quantised output's amax exchange)
        bool ok = true;
        for (int t = pair_id; ok && t < num_tiles; t += num_pairs) {
            const PairTile ti = pair_tile(t, rows_p, n_blocks, pM, player, list, meta, rank);
            const int m = ti.m_cta + r;                            // global row of A / D
            bool row_ok = r < ti.rows;
            if (player == DG_LAYOUT_CONTIGUOUS && row_ok) {
                const int gr = __ldg(meta + m);
                if (gr != ti.g) {
                    if (gr >= 0)
                        raise_status(status, DG_DEVFLAG_MIXED_BLOCK);
                    row_ok = false;
                }
            }
            const bool row_in = m < pM;
            const float *sfa_row = sfa + m;
            const int nb = min((ti.n0 + c0) >> 7, NBs - 1);
            const float *sfb_row = sfb + (static_cast<size_t>(ti.g) * NBs + nb) * KB;
            // The scales of a stage's two K blocks are copied into the warp's
            // shared memory one stage ahead (cp.async: nothing held in
            // registers, no TMA copy): lane i fetches sfa of its own row, lane
            // 0 also the two sfb values.  Buffer (par, kk): sfa at
            // [par][kk][lane], sfb at [par][64 + kk].
            auto prefetch = [&](int j, uint32_t par) {
                const uint32_t buf = scale_u32 + par * ((2 * 32 + 4) * 4);
#pragma unroll
                for (int kk = 0; kk < kPKps; ++kk) {
                    const int kb = j * kPKps + kk;
                    const bool in = row_in && kb < KB;
                    cp_async4(buf + (kk * 32 + lane) * 4, in ? sfa_row + static_cast<size_t>(kb) * pldsfa : sfa,
                              in ? 4u : 0u);
                    if (lane == 0)
                        cp_async4(buf + (64 + kk) * 4, kb < KB ? sfb_row + kb : sfb, kb < KB ? 4u : 0u);
                }
                cp_async_commit();
            };
            prefetch(0, 0);
            float2 acc[kPEpiCols / 2];
#pragma unroll
            for (int j = 0; j < kPEpiCols / 2; ++j)
                acc[j] = make_float2(0.0f, 0.0f);
            for (int j = 0; j < nst; ++j, ++gs) {
                const uint32_t par = static_cast<uint32_t>(j & 1);
                __syncwarp();                   // every lane is done reading the other buffer
                prefetch(j + 1, par ^ 1u);      // past the last stage: zero-size copies
                cp_async_wait<1>();             // this stage's scales have landed
                __syncwarp();                   // lane 0's sfb copies are visible to the warp
                const uint32_t buf = scale_u32 + par * ((2 * 32 + 4) * 4);
#pragma unroll
                for (int i = 0; i < kPKps; ++i) {
                    // fp32 product of the two scales, rounded once
                    const float sc = ld_shared_f32(buf + (i * 32 + lane) * 4) * ld_shared_f32(buf + (64 + i) * 4);
                    const float2 s2 = make_float2(sc, sc);
                    // every lane polls and the warp votes on each test, so
                    // that it leaves the wait converged for the warp-wide TMEM
                    // loads (cheaper than one poller and a broadcast, and than
                    // lanes that leave one by one)
                    if (!wait_phase_warp(tfull_bar(i), gs & 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t t_buf = t_lane + i * kPBN;
                    // The slot is released once all four 16-column loads have
                    // completed; the FMAs of the first two run while the last
                    // two are in flight (a wait covers every load the thread
                    // has issued, so the registers of a consumed chunk take
                    // the next one).
                    uint32_t v[16], w[16];
                    tmem_ld16(t_buf, v);
                    tmem_ld16(t_buf + 16, w);
                    tmem_wait_ld16(v);
                    tmem_wait_ld16(w);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        acc[k] = ffma2(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), s2, acc[k]);
                    tmem_ld16(t_buf + 32, v);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        acc[8 + k] =
                            ffma2(make_float2(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1])), s2, acc[8 + k]);
                    tmem_ld16(t_buf + 48, w);
                    tmem_wait_ld16(v);
                    tmem_wait_ld16(w);
                    tc_fence_before();
                    if (lane == 0)
                        mbar_arrive_cluster(tempty0 + 8u * i);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        acc[16 + k] =
                            ffma2(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), s2, acc[16 + k]);
                        acc[24 + k] =
                            ffma2(make_float2(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1])), s2, acc[24 + k]);
                    }
                }
                if (!ok)
                    break;
            }
            cp_async_wait<0>();
            if (!ok)
                break;
            if constexpr (!QOUT) {
                // bf16 first: the 64 accumulators become 32 packed words
                uint32_t pk[kPEpiCols / 2];
#pragma unroll
                for (int k = 0; k < kPEpiCols / 2; ++k)
                    pk[k] = pack_bf16x2(acc[k].x, acc[k].y);
                const uint32_t rows_ok = __ballot_sync(0xffffffffu, row_ok);
                const int cols_left = pN - (ti.n0 + c0);
                // The warp's 32 rows x 64 columns go into its staging rows in the
                // 128-byte swizzled order (chunk c of row r at c ^ (r & 7): the
                // lanes' 16-byte writes fall in distinct banks).  When all 32 rows
                // are stored, one TMA store writes them (clipped at the M and N
                // edges) and the warp moves on; otherwise (contiguous padding
                // rows, a rank with no rows) the warp stores the rows it owns.
                if (lane == 0)
                    bulk_wait_group_read0();        // the previous tile's store has read the staging rows
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(stage_u32 + lane * 128 + 16 * (c ^ (lane & 7)), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                                 pk[4 * c + 3]);
                if (rows_ok == 0xFFFFFFFFu && cols_left > 0) {
                    fence_proxy_async_smem();       // the writes above, visible to the TMA engine
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmap_d, stage_u32, ti.n0 + c0, ti.m_cta + q * 32);
                        bulk_commit_group();
                    }
                } else {
                    __syncwarp();
                    uint16_t *const d_warp = d + static_cast<size_t>(ti.m_cta + q * 32) * pN + ti.n0 + c0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = i * 4 + (lane >> 3);
                        const int cc = lane & 7;
                        if (((rows_ok >> rr) & 1u) && cc * 8 < cols_left) {
                            const uint4 v = ld_shared_v4(stage_u32 + rr * 128 + 16 * (cc ^ (rr & 7)));
                            st_global_v4(d_warp + static_cast<size_t>(rr) * pN + cc * 8, v.x, v.y, v.z, v.w);
                        }
                    }
                }
            } else {
                // Re-quantised output.  The row's 64 values, rounded to bf16,
                // give this slice's amax; the two slices of a 128-column group
                // (column slices 2h and 2h + 1 of the same lane quarter) meet
                // at xchg_bar(q, h), one phase per tile, and take the larger.
                // Then the scale s = max(amax, 1e-4) / 448 (IEEE division),
                // the codes E4M3(v / s) by the corrected reciprocal, staged in
                // 64-byte swizzled rows and stored row segment by row segment.
                auto unpack = [](uint32_t w) {
                    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
                };
                uint32_t pk[kPEpiCols / 2];
                float mx = 0.0f;
#pragma unroll
                for (int k = 0; k < kPEpiCols / 2; ++k) {
                    pk[k] = pack_bf16x2(acc[k].x, acc[k].y);
                    const float2 v = unpack(pk[k]);
                    mx = fmaxf(mx, fmaxf(fabsf(v.x), fabsf(v.y)));
                }
                const int h = grp >> 1;
                float *const amax_x = reinterpret_cast<float *>(smem + L::kAmaxOff) +
                                      tile_par * (kPBN / kPEpiCols) * kPRowsCta;
                amax_x[grp * kPRowsCta + r] = mx;
                mbar_arrive(xchg_bar(q, h));
                if (!wait_phase_warp(xchg_bar(q, h), tile_par, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const float amax = fmaxf(mx, amax_x[(grp ^ 1) * kPRowsCta + r]);
                const float sc = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
                const float rsc = __frcp_rn(sc);
                const uint32_t rows_ok = __ballot_sync(0xffffffffu, row_ok);
                const int cols_left = pN - (ti.n0 + c0);
                // 32 rows x 64 codes: chunk c (16 bytes) of row rr at c ^ ((rr >> 1) & 3)
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t wd[4];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float2 v0 = div2_rn(unpack(pk[8 * c + 4 * k + 0]), sc, rsc);
                        const float2 v1 = div2_rn(unpack(pk[8 * c + 4 * k + 1]), sc, rsc);
                        const float2 v2 = div2_rn(unpack(pk[8 * c + 4 * k + 2]), sc, rsc);
                        const float2 v3 = div2_rn(unpack(pk[8 * c + 4 * k + 3]), sc, rsc);
                        wd[2 * k] = e4m3x4(v0.x, v0.y, v1.x, v1.y);
                        wd[2 * k + 1] = e4m3x4(v2.x, v2.y, v3.x, v3.y);
                    }
                    st_shared_v4(stage_u32 + lane * 64 + 16 * (c ^ ((lane >> 1) & 3)), wd[0], wd[1], wd[2], wd[3]);
                }
                __syncwarp();
                if (cols_left > 0) {
                    uint8_t *const q_warp = qout + static_cast<size_t>(ti.m_cta + q * 32) * pN + ti.n0 + c0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = i * 8 + (lane >> 2);
                        const int cc = lane & 3;
                        if ((rows_ok >> rr) & 1u) {
                            const uint4 v = ld_shared_v4(stage_u32 + rr * 64 + 16 * (cc ^ ((rr >> 1) & 3)));
                            st_global_v4(q_warp + static_cast<size_t>(rr) * pN + cc * 16, v.x, v.y, v.z, v.w);
                        }
                    }
                    // one scale per row and 128-column group, M-major like sfa
                    if ((grp & 1) == 0 && row_ok)
                        sfo[static_cast<size_t>((ti.n0 >> 7) + h) * pldsfa + m] = sc;
                }
                __syncwarp();
                tile_par ^= 1u;
            }
        }
        // every bulk store of this thread has completed before the CTA ends
        if (lane == 0)
            bulk_wait_group0();
    }

    // ------------------------------------------------------------- teardown
    // Reconverge each warp (lane 0 of warps 0-3 ran its role alone), then meet
    // the peer CTA: neither CTA leaves while the other may still signal its
    // barriers or read its tensor memory.
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kPTmemCols);
    }
}

}  // namespace

bool pair_plan_ok(int layout, int M, int N, int K, int G, int num_sms)
{
    (void)G;
    (void)N;
    (void)K;
    if (num_sms < 2)
        return false;
    if (layout == DG_LAYOUT_DENSE)
        return true;
    if (layout == DG_LAYOUT_CONTIGUOUS)
        return M / kPRowsCta <= kPairMaxRows;
    return false;
}

int pair_smem_bytes()
{
    return PairSmem::kAlloc;
}

int pair_num_tiles(int layout, int M, int N, int G)
{
    // dense: exact; contiguous: an upper bound (one pair row per two blocks,
    // plus one per expert whose blocks do not pair up)
    const int n_blocks = ceil_div(N, kPBN);
    const int rows_p = layout == DG_LAYOUT_DENSE ? ceil_div(M, 2 * kPRowsCta)
                                                 : min(M / kPRowsCta, ceil_div(M / kPRowsCta, 2) + G);
    return rows_p * n_blocks;
}

dg_status_t launch_pair(int layout, const uint8_t *a, const float *sfa, const uint8_t *b, const float *sfb, uint16_t *d,
                        uint8_t *qout, float *sfo, const int32_t *meta, int M, int N, int K, int G,
                        int num_tiles_hint, void *stream, const DeviceInfo &info)
{
    const uint64_t KB = static_cast<uint64_t>(K / 128);
    CUtensorMap ta, tb;
    dg_status_t st;
    {
        // A: E4M3 [M][K] viewed as [K/128][M][128 B]; box: 2 K blocks x 128 rows
        const uint64_t dims[3] = {128, static_cast<uint64_t>(M), KB};
        const uint64_t strides[2] = {static_cast<uint64_t>(K), 128};
        const uint32_t box[3] = {128, kPRowsCta, kPKps};
        st = encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    {
        // B: E4M3 [N][K] (dense) or [G][N][K]; box: 2 K blocks x 128 rows
        const uint64_t dims[4] = {128, static_cast<uint64_t>(N), KB, static_cast<uint64_t>(G)};
        const uint64_t strides[3] = {static_cast<uint64_t>(K), 128, static_cast<uint64_t>(K) * N};
        const uint32_t box[4] = {128, kPRowsCta, kPKps, 1};
        st = encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, layout == DG_LAYOUT_DENSE ? 3 : 4, b, dims, strides,
                               box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    CUtensorMap td{};
    if (d) {
        // D: bf16 [M][N]; box: 64 columns x 32 rows (one epilogue warp's part
        // of a tile), 128-byte swizzled like the staging rows.  The
        // re-quantised output has no bf16 D and never reads this map.
        const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
        const uint64_t strides[1] = {static_cast<uint64_t>(N) * 2};
        const uint32_t box[2] = {static_cast<uint32_t>(kPEpiCols), 32};
        st = encode_tensor_map(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    const bool qmode = qout != nullptr;
    auto kernel = qmode ? fp8_gemm_pair_kernel<true> : fp8_gemm_pair_kernel<false>;
    st = ensure_smem_attr(reinterpret_cast<const void *>(kernel), PairSmem::kAlloc);
    if (st != DG_OK)
        return st;
    const int max_pairs = info.sm_count / 2;
    const int pairs = layout == DG_LAYOUT_DENSE ? min(max_pairs, max(1, num_tiles_hint)) : max_pairs;
    PairProblem prob{M, N, K, G, layout, round_up(M, 4)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = PairSmem::kAlloc;
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
    if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, td, sfa, sfb, d, qout, sfo, meta, prob, info.status_word) !=
        cudaSuccess)
        return DG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

}  // namespace dg
