// FP8 (E4M3) GEMM with fine-grained scaling and two-level accumulation on the
// sm_103a tensor cores, for the dense, MoE-contiguous and MoE-masked layouts.
//
// What it computes ("DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库", 技术细节/两级累加技术
// and 功能特色/细粒度缩放功能): for every 128-wide K block kb the tensor cores form the
// block's partial product P_kb = A[:, kb] . B[:, kb]^T in fp32 in tensor memory,
// and the CUDA cores promote it,
//     acc[m,n] = fmaf(P_kb[m,n], sfa[kb][m] * sfb[n/128][kb], acc[m,n]),
// kb ascending; D = bf16_rn(acc).
//
// How (the page's 线程专业化技术 and 统一的计算任务调度系统, redone for GB300):
// a persistent kernel, one CTA per SM, in four roles:
//   warp 0      TMA producer: streams A[128 rows] and B[BN rows] (128-byte
//               swizzled) into an S-stage shared-memory ring; the tensor maps
//               view K as (128 bytes) x (K blocks), so one box carries the
//               KPS K blocks of a stage;
//   warp 2      allocates and frees the TMEM columns;
//   warps 1, 2  MMA issuers, taking alternate ring stages: one thread each
//               waits for the stage's TMEM slot and data, issues
//               4 x tcgen05.mma kind::f8f6f4 (128 x BN x 32) per K block, each
//               K block into its own BN columns of the slot (the first MMA with
//               accumulate off), then commits once to the slot's "full"
//               barrier and once to the stage's "empty" barrier; warp 1 also
//               builds the masked layout's per-expert tile prefix;
//   warps 4..   epilogue warpgroups, each owning EPI_COLS of the tile's
//               columns; a thread owns one output row (TMEM lane).  Per slot
//               every lane polls the slot's barrier, the warp loads its
//               partial rows from TMEM and releases the slot, then scales each
//               K block's row by sfa * sfb (read from global memory a few K
//               blocks ahead into fixed registers) and FMAs it into fp32
//               registers (two values per packed f32x2 instruction), K blocks
//               ascending; after the last block it converts to bf16, stages
//               the rows in shared memory and writes them with one TMA store
//               per warp (row by row where some rows must not be written).
// An mbarrier handoff costs a few hundred cycles, so handoffs are per stage
// and per TMEM slot, not per MMA.  Tiles are 128 x 192 (4 one-K-block stages,
// two TMEM slots, 512 threads) when the problem has at least a full wave of
// them, else 128 x 128 (5 one-block stages, four slots, 384 threads) or
// 128 x 96 (3 two-block stages, two slots of two K blocks, 512 threads),
// whichever fills the SMs better.  Tiles are visited in a grouped order
// (kGroupM m-blocks per band) so that the CTAs running at the same time share
// A and B tiles through L2.
//
// Every wait is bounded: after kWaitTimeoutCycles a role raises the CTA's abort
// flag and DG_DEVFLAG_TIMEOUT, the producer waits (bounded) for its own copies
// in flight, the MMA thread drains its MMAs, TMEM is freed and the CTA exits.
#include <stdlib.h>

#include <algorithm>

#include "dg_common.h"
#include "dg_ptx.cuh"
#include "dg_wait.cuh"

namespace dg {
namespace {

constexpr int kBM = 128;                   // rows per tile (tcgen05 M)
constexpr int kBK = 128;                   // K per stage = one promotion block = one 128-byte row
constexpr int kEpiWarp0 = 4;                        // warps 0-3: producer, two MMA issuers, spare
constexpr int kIssuers = 2;                         // MMA-issuing threads (warps 1 and 2)

// Threads of the CTA for a tile width: 4 warps + one epilogue warpgroup per
// EPI_COLS columns (BN = 96: 3 x 32 columns, 512 threads; BN = 128: 2 x 64,
// 384 threads, 168 registers each; BN = 192: 3 x 64, 512 threads, 128).
template <int BN, int EPI_COLS>
struct Roles {
    static constexpr int kEpiGroups = BN / EPI_COLS;
    static constexpr int kNumEpiWarps = 4 * kEpiGroups;
    static constexpr int kThreads = 32 * (kEpiWarp0 + kNumEpiWarps);
};
constexpr int kGroupM = 16;                // m-blocks per rasterisation band
constexpr int kMaxBufs = 5;                // TMEM partial buffers at most (512 columns / BN)
constexpr int kMaxMaskedGroups = 1024;     // G limit of the masked layout (tile prefix in smem)

template <int BN, int STAGES, int EPI_COLS, int KPS>
struct SmemLayout {
    // one ring stage holds KPS consecutive K blocks of A and of B, each a
    // 128-byte-swizzled [rows][128] tile
    static constexpr int kASub = kBM * kBK;         // 16 KiB
    static constexpr int kBSub = BN * kBK;
    static constexpr int kABytes = KPS * kASub;
    static constexpr int kBBytes = KPS * kBSub;
    static constexpr int kAOff = 0;
    static constexpr int kBOff = kAOff + STAGES * kABytes;
    // output staging: each epilogue warp owns 32 rows x EPI_COLS bf16.  The
    // bf16 store uses the first 32 x 2 EPI_COLS bytes in its TMA store's
    // swizzled order; the re-quantised output pads its rows by 16 bytes so
    // that row-per-thread 16-byte writes do not collide on shared-memory banks
    static constexpr int kOutRowStride = EPI_COLS * 2 + 16;
    static constexpr int kOutWarpBytes = 32 * kOutRowStride;
    static constexpr int kOutOff = kBOff + STAGES * kBBytes;
    static constexpr int kBarOff = kOutOff + (BN / EPI_COLS) * 4 * kOutWarpBytes;
    // full[S], empty[S], tfull[kMaxBufs], tempty[kMaxBufs], drain[2], xchg[4]
    static constexpr int kNumBars = 2 * STAGES + 2 * kMaxBufs + 2 + 4;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // tmem base, abort flag
    static constexpr int kPrefixOff = kMiscOff + 16;
    // re-quantised output: per-row amax halves exchanged between the two
    // warpgroups of a 128-column group, double-buffered by tile parity
    static constexpr int kAmaxOff = kPrefixOff + (kMaxMaskedGroups + 1) * 4;
    static constexpr int kBytes = kAmaxOff + 2 * 2 * kBM * 4;
    static constexpr int kAlloc = kBytes + 1024;   // slack to align the base to 1024
};

struct Problem {
    int M;        // dense: rows; contiguous: sum_M; masked: max_m
    int N;
    int K;
    int G;
    int layout;
    int ldsfa;    // row stride of SFA (round_up(M, 4))
};

struct TileInfo {
    int g;
    int m0;        // first row of the tile within its expert's rows
    int n0;
    int rows;      // rows of the tile that are inside the problem
    bool skip;
};

template <int BN>
struct Sched {
    int m_blocks;     // dense / contiguous: m-blocks of the whole problem
    int n_blocks;
    int num_tiles;
    const int *prefix;   // masked: tile prefix per expert (smem)
    int G;

    __device__ __forceinline__ TileInfo tile(int t, const Problem &p, const int32_t *meta) const
    {
        TileInfo ti;
        ti.skip = false;
        if (p.layout == DG_LAYOUT_MASKED) {
            int lo = 0, hi = G;   // find g with prefix[g] <= t < prefix[g+1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] <= t)
                    lo = mid;
                else
                    hi = mid;
            }
            const int g = lo;
            const int local = t - prefix[g];
            const int valid = (prefix[g + 1] - prefix[g]) / n_blocks;   // m-blocks of expert g
            const int mb = local % valid;
            const int nb = local / valid;
            int mm = meta[g];
            mm = mm < 0 ? 0 : (mm > p.M ? p.M : mm);
            ti.g = g;
            ti.m0 = mb * kBM;
            ti.n0 = nb * BN;
            ti.rows = min(kBM, mm - ti.m0);
            return ti;
        }
        // grouped rasterisation: bands of kGroupM m-blocks, m fastest inside a band
        const int band_tiles = kGroupM * n_blocks;
        const int band = t / band_tiles;
        const int first_m = band * kGroupM;
        const int band_m = min(m_blocks - first_m, kGroupM);
        const int local = t - band * band_tiles;
        const int mb = first_m + local % band_m;
        const int nb = local / band_m;
        ti.m0 = mb * kBM;
        ti.n0 = nb * BN;
        ti.rows = min(kBM, p.M - ti.m0);
        ti.g = 0;
        if (p.layout == DG_LAYOUT_CONTIGUOUS) {
            const int g = meta[ti.m0];
            ti.g = g;
            ti.skip = (g < 0 || g >= p.G);
        }
        return ti;
    }
};

// Register cap per thread: at 128 x 96 (the small-M tile) 112, without
// spills, so that a CTA (512 threads) leaves 8k registers of the SM free:
// room for one block of the activation quantiser (8 warps x 32 registers),
// so that the GEMM launched behind it starts on an SM where one block is
// still running.  The other tiles take what their launch bounds allow.
template <int BN>
constexpr int max_regs()
{
    return BN == 96 ? 112 : 168;
}

// QOUT: instead of bf16 D, write D re-quantised as the next GEMM's activation
// operand: E4M3 codes qout (D's layout, one byte per element) and one fp32
// scale per 1x128 group of each row, sfo [(G,) N/128][ldsfa] (M-major), each
// group's scale and codes computed from the bf16-rounded values exactly as
// the 1x128 quantiser does.  Needs 128-column groups inside one tile (BN =
// 128, two 64-column warpgroups).
template <int BN, int STAGES, int EPI_COLS, int KPS, bool QOUT>
__global__ void __launch_bounds__(Roles<BN, EPI_COLS>::kThreads, 1) __maxnreg__(max_regs<BN>())
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const float *__restrict__ sfa, const float *__restrict__ sfb,
                    uint16_t *__restrict__ d, uint8_t *__restrict__ qout, float *__restrict__ sfo,
                    const int32_t *__restrict__ meta, Problem p, unsigned int *status)
{
    using L = SmemLayout<BN, STAGES, EPI_COLS, KPS>;
    static_assert(!QOUT || (BN == 128 && EPI_COLS == 64), "re-quantised output needs one 128-column group per tile");
    static_assert(QOUT || ((EPI_COLS == 32 || EPI_COLS == 64) && L::kOutOff % 1024 == 0 &&
                           L::kOutWarpBytes >= 32 * EPI_COLS * 2),
                  "bf16 output: each warp stages 32 rows x EPI_COLS on a swizzle-aligned boundary for its TMA store");
    constexpr int kNumEpiWarps = Roles<BN, EPI_COLS>::kNumEpiWarps;
    // TMEM slots: one per ring stage in flight between the MMAs and the
    // epilogue, each holding the KPS partial products (128 x BN fp32) of one
    // stage's K blocks; as many as fit in 512 columns.  A barrier handoff costs
    // a few hundred cycles, so the MMA side signals, and the epilogue releases,
    // a whole stage at once.
    constexpr int kSlotCols = KPS * BN;
    constexpr int kBufs = (512 / kSlotCols < kMaxBufs) ? 512 / kSlotCols : kMaxBufs;
    constexpr uint32_t kTmemCols = (kBufs * kSlotCols <= 32)    ? 32
                                   : (kBufs * kSlotCols <= 64)  ? 64
                                   : (kBufs * kSlotCols <= 128) ? 128
                                   : (kBufs * kSlotCols <= 256) ? 256
                                                                : 512;
    constexpr int kCols = EPI_COLS;                    // columns per epilogue warpgroup
    // TMEM loads of 32 columns (32x32b.x32): one per 32 columns of a K block.
    // Where registers allow, the next chunk's load overlaps this chunk's FMAs;
    // at BN = 192 (512 threads, 128 registers) one chunk is held at a time.
    constexpr int kW = 32;
    constexpr bool kPrefetchChunk = (BN != 192);
    constexpr int kChunks = kCols / kW;                // TMEM loads per K block
    constexpr uint32_t kStageTx = L::kABytes + L::kBBytes;
    constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, BN);
    static_assert(BN % EPI_COLS == 0 && EPI_COLS % kW == 0 && BN <= 256, "BN must be a multiple of EPI_COLS up to 256");
    static_assert(128 % kCols == 0, "the columns of one epilogue warpgroup must lie in one 128-column scale block");
    static_assert(kBufs >= 2, "at least two TMEM slots");
    // issuers alternate stages, so slot s is always written by issuer s % 2 and
    // each thread waits only for its own slot's previous release
    static_assert(kBufs % kIssuers == 0, "each TMEM slot must belong to one issuer");
    // the issuers test a stage's full barrier by parity only: waiting for the
    // TMEM slot's previous release first guarantees that every fill up to
    // (this use - STAGES) has been consumed only while slots <= stages
    static_assert(STAGES >= kBufs, "full-barrier parity test needs TMEM slots <= ring stages");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + kMaxBufs + b); };
    auto drain_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * kMaxBufs + i); };
    // re-quantised output: the two warps holding rows 32q..32q+31 meet here
    auto xchg_bar = [&](int q) { return bar0 + 8u * (2 * STAGES + 2 * kMaxBufs + 2 + q); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::kMiscOff + 4);
    int *prefix = reinterpret_cast<int *>(smem + L::kPrefixOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int KB = p.K / kBK;
    const int KP = (KB + KPS - 1) / KPS;   // ring stages (load units) per tile
    const int NBs = (p.N + 127) / 128;   // 128-column scale blocks of B

    // ------------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kNumEpiWarps);
        }
        for (int i = 0; i < kIssuers; ++i)
            mbar_init(drain_bar(i), 1);
        if constexpr (QOUT)
            for (int i = 0; i < 4; ++i)
                mbar_init(xchg_bar(i), 64);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 2) {
        // TMEM is allocated by warp 2 while thread 0 sets up the barriers
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    Sched<BN> sch;
    sch.n_blocks = (p.N + BN - 1) / BN;
    sch.G = p.G;
    sch.prefix = prefix;
    sch.m_blocks = (p.layout == DG_LAYOUT_MASKED) ? 0 : (p.M + kBM - 1) / kBM;
    sch.num_tiles = sch.m_blocks * sch.n_blocks;   // masked: set from the prefix below

    // TMA producer state (thread 0): a cursor over this CTA's (tile, K block)
    // load units and the ring position
    int p_stage = 0;
    uint32_t p_phase = 0;
    uint32_t pending = 0;        // stages with a copy whose consumption was not yet observed
    uint32_t pending_par = 0;    // full-barrier parity of each pending copy
    int p_t = blockIdx.x;
    int p_u = 0;                 // load unit (group of KPS K blocks) within the tile
    bool p_have = false;
    TileInfo p_ti{};
    // moves the cursor to the next unit to load; false when there is none
    auto p_next = [&]() -> bool {
        for (;;) {
            if (!p_have) {
                if (p_t >= sch.num_tiles)
                    return false;
                p_ti = sch.tile(p_t, p, meta);
                if (p_ti.skip) {
                    p_t += gridDim.x;
                    continue;
                }
                p_have = true;
                p_u = 0;
            }
            if (p_u < KP)
                return true;
            p_have = false;
            p_t += gridDim.x;
        }
    };
    // dense: stages of the first tile whose B copy (with the stage's
    // expect-tx) went out before the previous kernel had finished; only
    // their A copy is left to issue
    int p_pre = 0;
    // issues the loads of the unit under the cursor into the current stage
    auto p_issue = [&]() {
        const uint32_t fb = full_bar(p_stage);
        const uint32_t a_dst = sbase + L::kAOff + p_stage * L::kABytes;
        const uint32_t b_dst = sbase + L::kBOff + p_stage * L::kBBytes;
        // tensor maps view K as (128 bytes) x (K blocks); a box covers KPS
        // K blocks (past the last one it is zero-filled)
        const int kb0 = p_u * KPS;
        if (p_pre > 0) {
            --p_pre;
            tma_load_3d(a_dst, &tmap_a, fb, 0, p_ti.m0, kb0);
        } else if (p.layout == DG_LAYOUT_DENSE) {
            mbar_arrive_expect_tx(fb, kStageTx);
            tma_load_3d(a_dst, &tmap_a, fb, 0, p_ti.m0, kb0);
            tma_load_3d(b_dst, &tmap_b, fb, 0, p_ti.n0, kb0);
        } else if (p.layout == DG_LAYOUT_CONTIGUOUS) {
            mbar_arrive_expect_tx(fb, kStageTx);
            tma_load_3d(a_dst, &tmap_a, fb, 0, p_ti.m0, kb0);
            tma_load_4d(b_dst, &tmap_b, fb, 0, p_ti.n0, kb0, p_ti.g);
        } else {
            mbar_arrive_expect_tx(fb, kStageTx);
            tma_load_4d(a_dst, &tmap_a, fb, 0, p_ti.m0, kb0, p_ti.g);
            tma_load_4d(b_dst, &tmap_b, fb, 0, p_ti.n0, kb0, p_ti.g);
        }
        pending |= 1u << p_stage;
        pending_par = (pending_par & ~(1u << p_stage)) | (p_phase << p_stage);
        ++p_u;
        if (++p_stage == STAGES) {
            p_stage = 0;
            p_phase ^= 1u;
        }
    };
    if (threadIdx.x == 0 && p.layout == DG_LAYOUT_DENSE && p_next()) {
        // B is the weights: never written by a kernel that lets its
        // dependents start early (the activation quantiser, the GEMMs), so
        // its first stages can be copied while the previous kernel of the
        // stream, typically the quantiser producing A, is still running
        p_pre = min(STAGES, KP);
        for (int s = 0; s < p_pre; ++s) {
            mbar_arrive_expect_tx(full_bar(s), kStageTx);
            tma_load_3d(sbase + L::kBOff + s * L::kBBytes, &tmap_b, full_bar(s), 0, p_ti.n0, s * KPS);
            pending |= 1u << s;   // parity 0: the ring's first round
        }
    }
    // the previous kernel in the stream may still be running until here
    griddep_wait();
    if (threadIdx.x == 0 && p.layout != DG_LAYOUT_MASKED) {
        // the ring is empty: issue the first stage before the CTA barrier, so
        // that its copies overlap the TMEM allocation and the other warps'
        // set-up.  Only one: the first copies issue slowly (cold descriptors),
        // and the MMA issuers wait at the barrier for this thread.
        if (p_next())
            p_issue();
    }

    if (p.layout == DG_LAYOUT_MASKED && warp == 1) {
        // per-expert tile counts from masked_m, read on the device
        const int max_mb = (p.M + kBM - 1) / kBM;
        int running = 0;
        for (int base = 0; base < p.G; base += 32) {
            const int g = base + lane;
            int cnt = 0;
            if (g < p.G) {
                int mm = meta[g];
                if (mm < 0 || mm > p.M) {
                    raise_status(status, DG_DEVFLAG_MASKED_M_CLAMPED);
                    mm = mm < 0 ? 0 : p.M;
                }
                cnt = min((mm + kBM - 1) / kBM, max_mb) * sch.n_blocks;
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (g < p.G)
                prefix[g + 1] = running + incl;
            running += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            prefix[0] = 0;
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    tc_fence_after();
    // a kernel launched after this one with programmatic serialisation (the
    // activation quantiser of the next step) may be placed now; it waits for
    // this grid to complete before touching memory
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    if (p.layout == DG_LAYOUT_MASKED)
        sch.num_tiles = prefix[p.G];
    const uint32_t tmem_base = *tmem_slot;
    if (warp < kEpiWarp0) {
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            while (p_next()) {
                if (!wait_phase(empty_bar(p_stage), p_phase ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                pending &= ~(1u << p_stage);
                p_issue();
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if (pending & (1u << s))
                        drain_wait(full_bar(s), (pending_par >> s) & 1u);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------ MMA issuers
        // Two threads in two warps take alternate ring stages (by a running
        // count over all tiles), so that one's barrier waits and commits
        // overlap the other's MMAs.
        if (lane == 0) {
            const uint32_t me = static_cast<uint32_t>(warp - 1);
            const uint64_t desc_a0 = smem_desc_sw128(sbase + L::kAOff);
            const uint64_t desc_b0 = smem_desc_sw128(sbase + L::kBOff);
            uint32_t gu = 0;       // load units over all tiles: the ring position
            bool ok = true;
            for (int t = blockIdx.x; ok && t < sch.num_tiles; t += gridDim.x) {
                const TileInfo ti = sch.tile(t, p, meta);
                if (ti.skip)
                    continue;
                for (int u = 0; ok && u < KP; ++u, ++gu) {
                    if ((gu % kIssuers) != me)
                        continue;
                    const uint32_t stage = gu % STAGES;
                    const uint32_t phase = (gu / STAGES) & 1u;
                    const uint32_t slot = gu % kBufs;
                    const uint32_t sph = (gu / kBufs) & 1u;
                    const int kb0 = u * KPS;
                    const int nkb = min(KPS, KB - kb0);
                    // The slot first, then the data.  A stage's previous use may
                    // belong to the other issuer; once the epilogue has released
                    // this slot's previous use, every earlier stage has been
                    // consumed, so the full barrier cannot be two phases behind
                    // (a parity test could not tell those apart).
                    if (!wait_phase(tempty_bar(slot), sph ^ 1u, abort_flag, status) ||
                        !wait_phase(full_bar(stage), phase, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int j = 0; j < nkb; ++j) {
                        const uint64_t da = desc_a0 + static_cast<uint64_t>((stage * L::kABytes + j * L::kASub) >> 4);
                        const uint64_t db = desc_b0 + static_cast<uint64_t>((stage * L::kBBytes + j * L::kBSub) >> 4);
                        // each K block's partial product has its own BN columns of the slot
                        const uint32_t d_tmem = tmem_base + slot * kSlotCols + j * BN;
                        // 4 MMAs of K = 32 bytes; each step advances the start address by 32 B
                        mma_f8f6f4<false>(d_tmem, da, db, kIdesc);
                        mma_f8f6f4<true>(d_tmem, da + 2, db + 2, kIdesc);
                        mma_f8f6f4<true>(d_tmem, da + 4, db + 4, kIdesc);
                        mma_f8f6f4<true>(d_tmem, da + 6, db + 6, kIdesc);
                    }
                    mma_commit(tfull_bar(slot));
                    mma_commit(empty_bar(stage));
                }
            }
            // every MMA this thread issued has completed once this barrier flips
            mma_commit(drain_bar(me));
            drain_wait(drain_bar(me), 0);
        }
    }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const int grp = (warp - kEpiWarp0) >> 2;         // column slice of this warpgroup
        const int r = q * 32 + lane;                     // row of the tile owned by this thread
        const int c0 = grp * kCols;                      // first column of this warpgroup
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c0;
        int buf = 0;
        uint32_t tph = 0;
        bool ok = true;
        uint32_t tile_par = 0;   // alternates per tile done (QOUT's amax exchange buffer)
        for (int t = blockIdx.x; ok && t < sch.num_tiles; t += gridDim.x) {
            const TileInfo ti = sch.tile(t, p, meta);
            if (ti.skip) {
                if (ti.g >= p.G && threadIdx.x == kEpiWarp0 * 32)
                    raise_status(status, DG_DEVFLAG_BAD_EXPERT);
                continue;
            }
            // where this thread's row goes, and whether it is written at all
            bool row_ok = r < ti.rows;
            size_t d_row = 0;
            if (p.layout == DG_LAYOUT_MASKED) {
                d_row = static_cast<size_t>(ti.g) * p.M + ti.m0 + r;
            } else {
                d_row = static_cast<size_t>(ti.m0) + r;
                if (p.layout == DG_LAYOUT_CONTIGUOUS && row_ok) {
                    const int gr = __ldg(meta + ti.m0 + r);
                    if (gr != ti.g) {
                        if (gr >= 0)
                            raise_status(status, DG_DEVFLAG_MIXED_BLOCK);
                        row_ok = false;
                    }
                }
            }
            // This row's activation scales sfa[kb][m] (masked: per expert) and
            // the scales sfb[nb][kb] of the 128-column block of B holding this
            // warpgroup's columns are read kAhead K blocks ahead into register
            // rings indexed by kb % kAhead.  The K loop is unrolled by kAhead,
            // so every ring slot is one fixed register, written by its load and
            // read kAhead blocks later: rotating the values through moves would
            // make each move wait for the load still in flight.
            constexpr int kAhead = (BN == 192) ? 2 : 4;   // 512 threads x 128 registers at 192
            static_assert(kAhead % KPS == 0, "the unrolled K loop must cover whole ring stages");
            const bool row_in = ti.m0 + r < p.M;   // rows outside A read nothing
            const float *sfa_row = sfa + (p.layout == DG_LAYOUT_MASKED ? static_cast<size_t>(ti.g) * KB * p.ldsfa : 0) +
                                   ti.m0 + r;
            const int nb = min((ti.n0 + c0) >> 7, NBs - 1);
            const float *sfb_row = sfb + (static_cast<size_t>(ti.g) * NBs + nb) * KB;
            auto load_sa = [&](int kb) -> float {
                return (row_in && kb < KB) ? __ldg(sfa_row + static_cast<size_t>(kb) * p.ldsfa) : 0.0f;
            };
            auto load_sb = [&](int kb) -> float { return kb < KB ? __ldg(sfb_row + kb) : 0.0f; };
            float sa_r[kAhead], sb_r[kAhead];
#pragma unroll
            for (int j = 0; j < kAhead; ++j) {
                sa_r[j] = load_sa(j);
                sb_r[j] = load_sb(j);
            }

            float2 acc[kCols / 2];
#pragma unroll
            for (int j = 0; j < kCols / 2; ++j)
                acc[j] = make_float2(0.0f, 0.0f);

            for (int kb0 = 0; ok && kb0 < KB; kb0 += kAhead) {
#pragma unroll
                for (int j = 0; j < kAhead; ++j) {
                    const int kb = kb0 + j;
                    if (kb >= KB)
                        break;
                    // fp32 product of the two scales, rounded once
                    const float s = sa_r[j] * sb_r[j];
                    const float2 s2 = make_float2(s, s);
                    sa_r[j] = load_sa(kb + kAhead);
                    sb_r[j] = load_sb(kb + kAhead);
                    const int jj = j % KPS;                       // K block within its ring stage
                    const bool last_of_slot = (jj == KPS - 1) || (kb == KB - 1);
                    if (jj == 0) {
                        // wait until the MMAs of this stage are complete: every
                        // lane polls (one test serves the warp; cheaper than one
                        // poller and a broadcast; a vote on every test measured
                        // slower here, unlike in the pair kernel).  No bar.sync /
                        // bar.warp.sync here: those order memory, which would
                        // make the scale loads issued ahead complete first.
                        if (!__all_sync(0xffffffffu, wait_phase(tfull_bar(buf), tph, abort_flag, status))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint32_t t_buf = t_lane + buf * kSlotCols + jj * BN;
                    uint32_t v0[kW], v1[kPrefetchChunk ? kW : 1];
                    auto ld = [&](uint32_t addr, uint32_t(&r)[kW]) { tmem_ld32(addr, r); };
                    auto wait = [&](uint32_t(&r)[kW]) { tmem_wait_ld32(r); };
                    if constexpr (kPrefetchChunk) {
                        ld(t_buf, v0);
                        wait(v0);
#pragma unroll
                        for (int c = 0; c < kChunks; ++c) {
                            uint32_t(&cur)[kW] = (c & 1) ? v1 : v0;
                            uint32_t(&nxt)[kW] = (c & 1) ? v0 : v1;
                            if (c + 1 < kChunks) {
                                ld(t_buf + (c + 1) * kW, nxt);
                            } else if (last_of_slot) {
                                tc_fence_before();
                                if (lane == 0)
                                    mbar_arrive(tempty_bar(buf));
                            }
#pragma unroll
                            for (int i = 0; i < kW / 2; ++i)
                                acc[c * (kW / 2) + i] =
                                    ffma2(make_float2(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), s2,
                                          acc[c * (kW / 2) + i]);
                            if (c + 1 < kChunks)
                                wait(nxt);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < kChunks; ++c) {
                            ld(t_buf + c * kW, v0);
                            wait(v0);
                            if (c + 1 == kChunks && last_of_slot) {
                                tc_fence_before();
                                if (lane == 0)
                                    mbar_arrive(tempty_bar(buf));
                            }
#pragma unroll
                            for (int i = 0; i < kW / 2; ++i)
                                acc[c * (kW / 2) + i] =
                                    ffma2(make_float2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1])), s2,
                                          acc[c * (kW / 2) + i]);
                        }
                    }
                    if (last_of_slot && ++buf == kBufs) {
                        buf = 0;
                        tph ^= 1u;
                    }
                }
            }
            if (!ok)
                break;
            // Store: each thread writes its row into the warp's staging rows,
            // then the warp writes 32 rows x kCols out row-major, so that one
            // instruction covers whole row segments.  Rows that must not be
            // written (edges, masked tails, padding) are skipped.
            if constexpr (!QOUT) {
                // Each warp stages its 32 rows x kCols bf16 (kRowB bytes a
                // row) in the swizzled order of the output's TMA store, so
                // that the lanes' 16-byte writes fall in distinct banks:
                // 16-byte chunk c of row r sits at c ^ (r & 7) in 128-byte
                // rows (64 columns, 128-byte swizzle) and at c ^ ((r >> 1) & 3)
                // in 64-byte rows (32 columns, 64-byte swizzle).  When all 32
                // rows are stored, one TMA store writes them (clipped at the N
                // edge) and the warp moves on; otherwise (edges, masked tails,
                // padding) the warp stores the rows it owns.
                constexpr int kRowB = kCols * 2;
                constexpr int kRowChunks = kRowB / 16;
                auto swz = [](int rr) { return kRowB == 128 ? (rr & 7) : ((rr >> 1) & 3); };
                const uint32_t st0 = smem_u32(smem + L::kOutOff) + (warp - kEpiWarp0) * (32 * kRowB);
                if (lane == 0)
                    bulk_wait_group_read0();      // the previous tile's store has read these rows
                __syncwarp();
#pragma unroll
                for (int c = 0; c < kRowChunks; ++c)
                    st_shared_v4(st0 + lane * kRowB + 16 * (c ^ swz(lane)), pack_bf16x2(acc[c * 4 + 0].x, acc[c * 4 + 0].y),
                                 pack_bf16x2(acc[c * 4 + 1].x, acc[c * 4 + 1].y),
                                 pack_bf16x2(acc[c * 4 + 2].x, acc[c * 4 + 2].y),
                                 pack_bf16x2(acc[c * 4 + 3].x, acc[c * 4 + 3].y));
                const uint32_t rows_ok = __ballot_sync(0xffffffffu, row_ok);
                const size_t warp_row0 = d_row - lane;           // D row of this warp's first row
                const int cols_left = p.N - (ti.n0 + c0);
                if (rows_ok == 0xFFFFFFFFu && cols_left > 0) {
                    fence_proxy_async_smem();     // the writes above, visible to the TMA engine
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmap_d, st0, ti.n0 + c0, static_cast<int>(warp_row0));
                        bulk_commit_group();
                    }
                } else {
                    __syncwarp();
                    constexpr int kRowsPerPass = 32 / kRowChunks;
#pragma unroll
                    for (int i = 0; i < kRowChunks; ++i) {
                        const int rr = i * kRowsPerPass + lane / kRowChunks;
                        const int cc = lane % kRowChunks;
                        if (((rows_ok >> rr) & 1u) && cc * 8 < cols_left) {
                            const uint4 v = ld_shared_v4(st0 + rr * kRowB + 16 * (cc ^ swz(rr)));
                            st_global_v4(d + (warp_row0 + rr) * p.N + ti.n0 + c0 + cc * 8, v.x, v.y, v.z, v.w);
                        }
                    }
                }
            } else {
                // Re-quantised output.  Each thread rounds its 64 values to
                // bf16, stages them in its row of the warp's shared-memory
                // rows (128 bytes) and takes their amax; the two warpgroups
                // hold the two 64-column halves of each row's 128-column
                // group, and the row's amax is the larger of the halves'.
                auto unpack = [](uint32_t w) {
                    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
                };
                uint8_t *const stage = smem + L::kOutOff + (warp - kEpiWarp0) * L::kOutWarpBytes;
                const uint32_t my_row = smem_u32(stage) + lane * L::kOutRowStride;
                float m = 0.0f;
#pragma unroll
                for (int c = 0; c < kCols / 8; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        w[k] = pack_bf16x2(acc[c * 4 + k].x, acc[c * 4 + k].y);
                        const float2 v = unpack(w[k]);
                        m = fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y)));
                    }
                    st_shared_v4(my_row + c * 16, w[0], w[1], w[2], w[3]);
                }
                float *const amax_x = reinterpret_cast<float *>(smem + L::kAmaxOff) + tile_par * 2 * kBM;
                amax_x[grp * kBM + r] = m;
                // the two warps holding these 32 rows meet at xchg_bar(q), one
                // phase per tile, with a bounded wait (a partner that gave up
                // on an earlier wait never arrives)
                mbar_arrive(xchg_bar(q));
                uint32_t met = 1;
                if (lane == 0)
                    met = wait_phase(xchg_bar(q), tile_par, abort_flag, status) ? 1u : 0u;
                if (__shfl_sync(0xffffffffu, met, 0) == 0) {
                    ok = false;
                    break;
                }
                __syncwarp();
                const float amax = fmaxf(m, amax_x[(grp ^ 1) * kBM + r]);
                const float sc = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
                const float rsc = __frcp_rn(sc);
                // 8 values (16 bytes of bf16) in, 8 codes out, written over
                // the front of the same row (behind what has been read)
#pragma unroll 2
                for (int c = 0; c < kCols / 8; ++c) {
                    const uint4 w = ld_shared_v4(my_row + c * 16);
                    const float2 v0 = div2_rn(unpack(w.x), sc, rsc);
                    const float2 v1 = div2_rn(unpack(w.y), sc, rsc);
                    const float2 v2 = div2_rn(unpack(w.z), sc, rsc);
                    const float2 v3 = div2_rn(unpack(w.w), sc, rsc);
                    st_shared_v2(my_row + c * 8, e4m3x4(v0.x, v0.y, v1.x, v1.y), e4m3x4(v2.x, v2.y, v3.x, v3.y));
                }
                __syncwarp();
                const uint32_t rows_ok = __ballot_sync(0xffffffffu, row_ok);
                const size_t warp_row0 = d_row - lane;
                constexpr int kChunksPerRow = kCols / 16;        // 16-byte chunks of codes per row
#pragma unroll
                for (int i = 0; i < kChunksPerRow; ++i) {
                    const int idx = i * 32 + lane;
                    const int rr = idx / kChunksPerRow;
                    const int cc = idx % kChunksPerRow;
                    const int col = ti.n0 + c0 + cc * 16;
                    if (((rows_ok >> rr) & 1u) && col < p.N) {
                        const uint4 v = ld_shared_v4(smem_u32(stage) + rr * L::kOutRowStride + cc * 16);
                        st_global_v4(qout + (warp_row0 + rr) * p.N + col, v.x, v.y, v.z, v.w);
                    }
                }
                if (grp == 0 && row_ok) {
                    // scales M-major: [(g,) n-group][row], the activation layout
                    const size_t ngroups = static_cast<size_t>(p.N) / 128;
                    const size_t srow = p.layout == DG_LAYOUT_MASKED ? static_cast<size_t>(ti.m0 + r) : d_row;
                    const size_t sgrp = (p.layout == DG_LAYOUT_MASKED ? static_cast<size_t>(ti.g) * ngroups : 0) +
                                        static_cast<size_t>(ti.n0 / 128);
                    sfo[sgrp * p.ldsfa + srow] = sc;
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
    // Lane 0 of warps 0-2 ran its role alone: reconverge each warp before the
    // CTA barrier (bar.sync is the aligned form, which expects every thread of
    // a warp to execute it together).
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ----------------------------------------------------------------- host side
struct Plan {
    int bm;       // 128, or 256 for the CTA-pair kernel
    int bn;
    int stages;
    int num_tiles;
    int grid;
    int smem;
};

// Tile configurations compiled in (width, stages, epilogue columns per
// warpgroup).  The plan takes 128 x 192 when the problem has at least one full
// wave of such tiles; otherwise the narrower width whose busiest CTA streams
// the fewest bytes: waves x (128 + BN) rows of operand per K block.  For
// M = 256, N = 7168 on 152 SMs that is BN = 96 (150 tiles, one wave) over
// BN = 128 (112 tiles), the pages' 112-versus-128 argument redone for this
// SM count.
struct TileCfg {
    int bn;
    int stages;     // ring stages
    int epi_cols;   // columns per epilogue warpgroup
    int kps;        // K blocks per ring stage (one TMA box per operand)
};
// A TMA copy costs its SM a slot of a few hundred cycles plus the bytes, so
// the 128 x 96 tile streams two K blocks per box (and hands them to the
// epilogue as one TMEM slot).  At 128 x 192 two-block stages leave room for
// two stages and TMEM for two one-block slots, which needs a single issuer:
// measured slower than four one-block stages with two issuers.
constexpr TileCfg kCfg96{96, 3, 32, 2};
constexpr TileCfg kCfg128{128, 5, 64, 1};
constexpr TileCfg kCfg192{192, 4, 64, 1};

int forced_bn()
{
    // DG_FORCE_BN=96|128|192 pins the tile width of the one-SM kernel, 256
    // the CTA-pair kernel (where the layout has one)
    const char *e = getenv("DG_FORCE_BN");
    const int b = e ? atoi(e) : 0;
    return (b == 96 || b == 128 || b == 192 || b == 256) ? b : 0;
}

int smem_for(int bn)
{
    return bn == 192 ? SmemLayout<192, kCfg192.stages, kCfg192.epi_cols, kCfg192.kps>::kAlloc
           : bn == 96 ? SmemLayout<96, kCfg96.stages, kCfg96.epi_cols, kCfg96.kps>::kAlloc
                      : SmemLayout<128, kCfg128.stages, kCfg128.epi_cols, kCfg128.kps>::kAlloc;
}

Plan make_plan(int layout, int M, int N, int K, int G, int num_sms, bool qout = false, int expected_m = 0)
{
    Plan pl;
    // The CTA-pair kernel (256 x 256 tiles on two SMs) when the problem fills
    // at least one wave of pairs and K is long enough (at least 16 K blocks)
    // to amortise a tile's ring fill and store: it takes in 63 bytes per SM
    // cycle at the FP8 tensor rate, which one SM's TMA can sustain, where the
    // one-SM tiles need 94-128.  Its 128-column scale groups lie inside a
    // tile, so it also writes the re-quantised output.
    int fb = forced_bn();
    if (qout && fb != 256 && fb != 128)
        fb = 0;
    if (pair_plan_ok(layout, M, N, K, G, num_sms) &&
        (fb == 256 || (fb == 0 && K >= 16 * kBK && pair_num_tiles(layout, M, N, G) >= num_sms / 2))) {
        pl.bm = 256;
        pl.bn = 256;
        pl.stages = 3;
        pl.smem = pair_smem_bytes();
        pl.num_tiles = pair_num_tiles(layout, M, N, G);
        pl.grid = layout == DG_LAYOUT_DENSE ? 2 * std::min(num_sms / 2, std::max(1, pl.num_tiles)) : 2 * (num_sms / 2);
        return pl;
    }
    (void)K;
    pl.bm = kBM;
    // masked: the m-blocks the typical expert fills (expected_m, the caller's
    // hint; 0 = every buffer full) decide the width; the grid is fixed and
    // the kernel walks the real tile count
    const int rows_g = (layout == DG_LAYOUT_MASKED && expected_m > 0) ? std::min(expected_m, M) : M;
    const int mblk = layout == DG_LAYOUT_MASKED ? G * ceil_div(rows_g, kBM) : ceil_div(M, kBM);
    // a re-quantised output needs each 128-column scale group inside one tile
    int bn = qout ? 128 : (fb == 256 ? 0 : fb);
    if (bn == 0) {
        if (static_cast<long long>(mblk) * ceil_div(N, 192) >= num_sms) {
            bn = 192;
        } else {
            long long best = -1;
            for (int cand : {128, 96}) {
                const long long tiles = static_cast<long long>(mblk) * ceil_div(N, cand);
                const long long waves = (tiles + num_sms - 1) / num_sms;
                const long long cost = waves * (kBM + cand);
                if (best < 0 || cost < best) {
                    best = cost;
                    bn = cand;
                }
            }
        }
    }
    pl.bn = bn;
    pl.stages = bn == 192 ? kCfg192.stages : bn == 96 ? kCfg96.stages : kCfg128.stages;
    pl.smem = smem_for(bn);
    pl.num_tiles = (layout == DG_LAYOUT_MASKED ? G * ceil_div(M, kBM) : mblk) * ceil_div(N, bn);
    if (layout == DG_LAYOUT_MASKED)
        pl.grid = num_sms;   // fixed: the real tile count is only known on the device
    else
        pl.grid = pl.num_tiles < num_sms ? pl.num_tiles : num_sms;
    if (pl.grid < 1)
        pl.grid = 1;
    return pl;
}

dg_status_t check_common(const void *a, const void *sfa, const void *b, const void *sfb, const void *d, int M,
                         int N, int K)
{
    if (!a || !sfa || !b || !sfb || !d || M <= 0 || N <= 0 || K <= 0)
        return DG_ERR_INVALID_ARG;
    if (K % kBK != 0 || N % 8 != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d))
        return DG_ERR_MISALIGNED;
    return DG_OK;
}

dg_status_t launch(int layout, const uint8_t *a, const float *sfa, const uint8_t *b, const float *sfb, uint16_t *d,
                   uint8_t *qout, float *sfo, const int32_t *meta, int M, int N, int K, int G, void *stream,
                   int expected_m = 0)
{
    DeviceInfo info;
    dg_status_t st = current_device(&info);
    if (st != DG_OK)
        return st;
    const bool qmode = qout != nullptr;
    const Plan pl = make_plan(layout, M, N, K, G, info.sm_count, qmode, expected_m);
    if (pl.bm == 256)
        return launch_pair(layout, a, sfa, b, sfb, d, qout, sfo, meta, M, N, K, G, pl.num_tiles, stream, info);
    const int ldsfa = round_up(M, 4);

    // Tensor maps view each K-major operand as [..][rows][K/128][128 bytes]:
    // dim 0 is the 128-byte row segment of one K block, dim 1 the row (stride
    // K), dim 2 the K block (stride 128) and dim 3, for the grouped operands,
    // the expert.  A box is 128 bytes x rows x KPS K blocks.
    const int kps = pl.bn == 192 ? kCfg192.kps : pl.bn == 96 ? kCfg96.kps : kCfg128.kps;
    const uint64_t KB = static_cast<uint64_t>(K / kBK);
    CUtensorMap ta, tb;
    {
        // A: E4M3 [rows][K] (dense / contiguous) or [G][max_m][K] (masked)
        const uint64_t dims[4] = {static_cast<uint64_t>(kBK), static_cast<uint64_t>(M), KB, static_cast<uint64_t>(G)};
        const uint64_t strides[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(kBK),
                                     static_cast<uint64_t>(K) * M};
        const uint32_t box[4] = {kBK, kBM, static_cast<uint32_t>(kps), 1};
        st = encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, layout == DG_LAYOUT_MASKED ? 4 : 3, a, dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    {
        // B: E4M3 [N][K] (dense) or [G][N][K]
        const uint64_t dims[4] = {static_cast<uint64_t>(kBK), static_cast<uint64_t>(N), KB, static_cast<uint64_t>(G)};
        const uint64_t strides[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(kBK),
                                     static_cast<uint64_t>(K) * N};
        const uint32_t box[4] = {kBK, static_cast<uint32_t>(pl.bn), static_cast<uint32_t>(kps), 1};
        st = encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, layout == DG_LAYOUT_DENSE ? 3 : 4, b, dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DG_OK)
            return st;
    }
    // D (bf16 output): [rows][N], masked [G x max_m][N]; box: one epilogue
    // warp's 32 rows x its columns (64 at 128-byte swizzle, 32 at 64-byte),
    // swizzled like its staging rows.  The re-quantised output has no bf16 D
    // and never reads this map.
    CUtensorMap td{};
    if (d) {
        const int epi_cols = pl.bn == 192 ? kCfg192.epi_cols : pl.bn == 96 ? kCfg96.epi_cols : kCfg128.epi_cols;
        const uint64_t rows = layout == DG_LAYOUT_MASKED ? static_cast<uint64_t>(G) * M : static_cast<uint64_t>(M);
        const uint64_t dims[2] = {static_cast<uint64_t>(N), rows};
        const uint64_t strides[1] = {static_cast<uint64_t>(N) * 2};
        const uint32_t box[2] = {static_cast<uint32_t>(epi_cols), 32};
        st = encode_tensor_map(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, dims, strides, box,
                               epi_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
        if (st != DG_OK)
            return st;
    }
    auto kernel = qmode         ? fp8_gemm_kernel<128, kCfg128.stages, kCfg128.epi_cols, kCfg128.kps, true>
                  : pl.bn == 192 ? fp8_gemm_kernel<192, kCfg192.stages, kCfg192.epi_cols, kCfg192.kps, false>
                  : pl.bn == 96  ? fp8_gemm_kernel<96, kCfg96.stages, kCfg96.epi_cols, kCfg96.kps, false>
                                 : fp8_gemm_kernel<128, kCfg128.stages, kCfg128.epi_cols, kCfg128.kps, false>;
    const int threads = pl.bn == 192  ? Roles<192, kCfg192.epi_cols>::kThreads
                        : pl.bn == 96 ? Roles<96, kCfg96.epi_cols>::kThreads
                                      : Roles<128, kCfg128.epi_cols>::kThreads;
    st = ensure_smem_attr(reinterpret_cast<const void *>(kernel), pl.smem);
    if (st != DG_OK)
        return st;
    Problem prob{M, N, K, G, layout, ldsfa};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, td, sfa, sfb, d, qout, sfo, meta, prob, info.status_word) !=
        cudaSuccess)
        return DG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

}  // namespace
}  // namespace dg

extern "C" dg_status_t dg_fp8_gemm_nt(const uint8_t *a, const float *sfa, const uint8_t *b, const float *sfb,
                                      uint16_t *d, int M, int N, int K, void *stream)
{
    dg_status_t st = dg::check_common(a, sfa, b, sfb, d, M, N, K);
    if (st != DG_OK)
        return st;
    return dg::launch(DG_LAYOUT_DENSE, a, sfa, b, sfb, d, nullptr, nullptr, nullptr, M, N, K, 1, stream);
}

extern "C" dg_status_t dg_fp8_grouped_contiguous(const uint8_t *a, const float *sfa, const uint8_t *b,
                                                 const float *sfb, uint16_t *d, const int32_t *m_indices,
                                                 int sum_M, int N, int K, int G, void *stream)
{
    dg_status_t st = dg::check_common(a, sfa, b, sfb, d, sum_M, N, K);
    if (st != DG_OK)
        return st;
    if (!m_indices || G <= 0)
        return DG_ERR_INVALID_ARG;
    if (sum_M % dg::kBM != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!dg::aligned16(m_indices))
        return DG_ERR_MISALIGNED;
    return dg::launch(DG_LAYOUT_CONTIGUOUS, a, sfa, b, sfb, d, nullptr, nullptr, m_indices, sum_M, N, K, G, stream);
}

extern "C" dg_status_t dg_fp8_grouped_masked(const uint8_t *a, const float *sfa, const uint8_t *b,
                                             const float *sfb, uint16_t *d, const int32_t *masked_m, int G,
                                             int max_m, int N, int K, int expected_m, void *stream)
{
    dg_status_t st = dg::check_common(a, sfa, b, sfb, d, max_m, N, K);
    if (st != DG_OK)
        return st;
    if (!masked_m || G <= 0)
        return DG_ERR_INVALID_ARG;
    if (G > dg::kMaxMaskedGroups)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!dg::aligned16(masked_m))
        return DG_ERR_MISALIGNED;
    return dg::launch(DG_LAYOUT_MASKED, a, sfa, b, sfb, d, nullptr, nullptr, masked_m, max_m, N, K, G, stream,
                      expected_m);
}

// ---------------------------------------- re-quantised output (E4M3 + 1x128)
namespace dg {
namespace {
dg_status_t check_qout(const uint8_t *q, const float *sfo, int N)
{
    if (!q || !sfo)
        return DG_ERR_INVALID_ARG;
    if (N % 128 != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(q) || !aligned16(sfo))
        return DG_ERR_MISALIGNED;
    return DG_OK;
}
}  // namespace
}  // namespace dg

extern "C" dg_status_t dg_fp8_gemm_nt_q(const uint8_t *a, const float *sfa, const uint8_t *b, const float *sfb,
                                        uint8_t *q, float *sfo, int M, int N, int K, void *stream)
{
    // the D check of check_common is made on q (its address and alignment)
    dg_status_t st = dg::check_common(a, sfa, b, sfb, q, M, N, K);
    if (st == DG_OK)
        st = dg::check_qout(q, sfo, N);
    if (st != DG_OK)
        return st;
    return dg::launch(DG_LAYOUT_DENSE, a, sfa, b, sfb, nullptr, q, sfo, nullptr, M, N, K, 1, stream);
}

extern "C" dg_status_t dg_fp8_grouped_contiguous_q(const uint8_t *a, const float *sfa, const uint8_t *b,
                                                   const float *sfb, uint8_t *q, float *sfo,
                                                   const int32_t *m_indices, int sum_M, int N, int K, int G,
                                                   void *stream)
{
    dg_status_t st = dg::check_common(a, sfa, b, sfb, q, sum_M, N, K);
    if (st == DG_OK)
        st = dg::check_qout(q, sfo, N);
    if (st != DG_OK)
        return st;
    if (!m_indices || G <= 0)
        return DG_ERR_INVALID_ARG;
    if (sum_M % dg::kBM != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!dg::aligned16(m_indices))
        return DG_ERR_MISALIGNED;
    return dg::launch(DG_LAYOUT_CONTIGUOUS, a, sfa, b, sfb, nullptr, q, sfo, m_indices, sum_M, N, K, G, stream);
}

extern "C" dg_status_t dg_fp8_grouped_masked_q(const uint8_t *a, const float *sfa, const uint8_t *b,
                                               const float *sfb, uint8_t *q, float *sfo, const int32_t *masked_m,
                                               int G, int max_m, int N, int K, int expected_m, void *stream)
{
    dg_status_t st = dg::check_common(a, sfa, b, sfb, q, max_m, N, K);
    if (st == DG_OK)
        st = dg::check_qout(q, sfo, N);
    if (st != DG_OK)
        return st;
    if (!masked_m || G <= 0)
        return DG_ERR_INVALID_ARG;
    if (G > dg::kMaxMaskedGroups)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (!dg::aligned16(masked_m))
        return DG_ERR_MISALIGNED;
    // expected_m only sizes the bf16 call's tiles; a re-quantised output
    // always takes 128 x 128 tiles, whatever the rows per expert
    return dg::launch(DG_LAYOUT_MASKED, a, sfa, b, sfb, nullptr, q, sfo, masked_m, max_m, N, K, G, stream);
}

extern "C" dg_status_t dg_query_plan(int layout, int M, int N, int K, int G, int expected_m, int num_sms,
                                     dg_plan_t *out)
{
    if (!out || M <= 0 || N <= 0 || K <= 0 || G <= 0 || expected_m < 0 ||
        (layout != DG_LAYOUT_DENSE && layout != DG_LAYOUT_CONTIGUOUS && layout != DG_LAYOUT_MASKED))
        return DG_ERR_INVALID_ARG;
    if (K % dg::kBK != 0 || N % 8 != 0)
        return DG_ERR_UNSUPPORTED_SHAPE;
    if (num_sms <= 0) {
        dg::DeviceInfo info;
        dg_status_t st = dg::current_device(&info);
        if (st != DG_OK)
            return st;
        num_sms = info.sm_count;
    }
    const dg::Plan pl = dg::make_plan(layout, M, N, K, G, num_sms, false, expected_m);
    out->block_m = pl.bm;
    out->block_n = pl.bn;
    out->stages = pl.stages;
    out->num_tiles = pl.num_tiles;
    out->grid = pl.grid;
    out->smem_bytes = pl.smem;
    return DG_OK;
}
