// gemm_rs.cu -- matmul followed by a ring reduce-scatter, fused on the
// 5th-generation tensor cores.
//
// Sources: "TPU 与分布式通信原语", section "collective matmul" (matmul-reduce-
// scatter: every rank multiplies its activations by its row shard of W2,
// casts the partial product to bf16, lays it out chunk-major by output
// columns and reduce-scatters it round the ring); "Triton-distributed 语义",
// section "GEMM + ReduceScatter 重叠" (the GEMM produces output tiles, the
// reduce-scatter consumes each tile as soon as it exists).
//
// On one GPU every rank's partial product of an output tile can be formed
// where it is consumed, so the reduce-scatter consumer is the GEMM's own
// epilogue and partial products never reach HBM.  The output tile (m, n)
// lies in column chunk k = n / (N/P); its value is the ring reduce-scatter's
//     R = ((C_{k+1} (+) C_{k+2}) (+) ...) (+) C_k,   C_r = bf16(A_r . B_r^T)
// with (+) the bf16 hop add (binary32 add, rounded to bf16) -- the order in
// which the ring of the same section folds chunk k.  The MMA warp computes
// the P partial tiles in that order into two alternating TMEM accumulators;
// the epilogue rounds each to bf16 and folds it into a register-resident
// bf16 tile, then writes the finished tile to out_k.
//
// One persistent launch, one 256-thread block per SM: warp 0 TMA producer
// (4-stage ring of 128x64 A and 256x64 B tiles, 128-byte swizzle), warp 1 MMA
// issuer (tcgen05.mma.cta_group::1.kind::f16, M=128, N=256, K=16), warp 2
// TMEM allocator (512 columns), warps 4-7 epilogue.  Every wait is bounded.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "gemm_cfg.h"
#include "tc.cuh"

namespace rc {
namespace grs {

using namespace tc;

// The odd CTA's epilogue tells the even CTA's MMA warp that it has read its
// half of an accumulator.  Those TMEM loads have completed (tcgen05.wait::ld)
// before the arrival and the arrival publishes nothing else, so it needs no
// release semantics: a relaxed arrival at cluster scope.  Measured on GB300
// (P=8, 8192x4096x512 per rank, an accumulator handed back every K=512):
// 0.1627-0.1630 ms with a release arrival, 0.1555-0.1560 ms relaxed.
__device__ __forceinline__ void arrive_remote_relaxed(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

constexpr int BM = 128, BN = 256, BK = 64, UK = 16;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;   // 16 KiB
constexpr int B_STAGE = BN * BK * 2;   // 32 KiB
constexpr int THREADS = 256;
constexpr int TMEM_COLS = 512;         // two 128x256 fp32 accumulators
constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

struct Params {
    char *out;
    size_t out_stride;
    WsHeader *hdr;
    int P, M, N, K;          // K: per-rank inner dimension
    int n_chunk;             // N / P columns per rank
    int m_tiles, n_tiles, total_tiles;
    int st32;                // 1: output rows start on 32-byte boundaries (full-sector stores)
    unsigned long long timeout_ns;
};

// Tile t -> (m block, n block); n-major within an m block keeps a tile row's
// A operands hot in L2.
// The reduced output, which nothing reads in the launch, is stored
// evict_first (1) so that it does not push operand rows out of L2; 0: normal.
#ifndef RC_GRS_OUT_POLICY
#define RC_GRS_OUT_POLICY 1
#endif
constexpr int OUT_POL = RC_GRS_OUT_POLICY ? kStEvictFirst : kStNormal;

__device__ __forceinline__ void tile_of(const Params &p, int t, int &m, int &n)
{
    m = t / p.n_tiles;
    n = t % p.n_tiles;
}

__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_rs(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = sA + STAGES * A_STAGE;
    uint8_t *bars_g = gbase + STAGES * (A_STAGE + B_STAGE);
    const uint32_t bars = smem_u32(bars_g);
    const uint32_t full_bar = bars, empty_bar = bars + 8 * STAGES;
    const uint32_t tfull_bar = bars + 16 * STAGES, tempty_bar = tfull_bar + 16;
    const uint32_t drain_bar = tempty_bar + 16;
    uint32_t *tmem_slot = (uint32_t *)(bars_g + 16 * STAGES + 40);
    int *abort_flag = (int *)(bars_g + 16 * STAGES + 44);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar + 8 * a, 1);
            mbar_init(tempty_bar + 8 * a, 4);   // one arrive per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_b) : "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Abort ab{abort_flag, p.hdr, p.timeout_ns, 0xA7u};
    const int ksteps = p.K / BK;
    const int P = p.P;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: for every tile, the P partial products in ring order
        uint32_t stage = 0, phase = 0;
        int issued[STAGES] = {0, 0, 0, 0};
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int m, n;
            tile_of(p, t, m, n);
            const int k = (n * BN) / p.n_chunk;
            for (int jj = 1; jj <= P && ok; ++jj) {
                const int r = (k + jj) % P;               // jj = P is rank k itself, folded last
                for (int kb = 0; kb < ksteps; ++kb) {
                    if (!wait_bar(empty_bar + 8 * stage, phase ^ 1u, ab, 2)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full_bar + 8 * stage, A_STAGE + B_STAGE);
                    tma_load_3d(sA + stage * A_STAGE, &map_a, kb * BK, m * BM, r, full_bar + 8 * stage);
                    tma_load_3d(sB + stage * B_STAGE, &map_b, kb * BK, n * BN, r, full_bar + 8 * stage);
                    issued[stage]++;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (*(volatile int *)abort_flag) {
            for (int s = 0; s < STAGES; ++s)
                if (issued[s] > 0) wait_bar(full_bar + 8 * s, (uint32_t)((issued[s] - 1) & 1), ab, 9, true);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer: one partial product per accumulator
        uint32_t stage = 0, phase = 0;
        int it = 0;     // partial products issued so far
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            for (int jj = 1; jj <= P; ++jj, ++it) {
                const uint32_t acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!wait_bar(tempty_bar + 8 * acc, acc_phase ^ 1u, ab, 3)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int kb = 0; kb < ksteps; ++kb) {
                    if (!wait_bar(full_bar + 8 * stage, phase, ab, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(sA + stage * A_STAGE);
                    const uint64_t bd = smem_desc_sw128(sB + stage * B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk)
                        tc_mma(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc, (kb | kk) != 0);
                    tc_commit(empty_bar + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit(tfull_bar + 8 * acc);
                if (!ok) break;
            }
        }
        tc_commit(drain_bar);
        wait_bar(drain_bar, 0, ab, 10, true);
    } else if (warp >= 4) {
        // ---------------- epilogue: round each partial to bf16 and fold it
        const int q = warp - 4;          // TMEM lane quadrant = tile rows q*32 .. q*32+31
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int m, n;
            tile_of(p, t, m, n);
            const int k = (n * BN) / p.n_chunk;
            uint32_t acc[BN / 2];        // the folded tile row: 256 bf16 as 128 packed pairs
            for (int jj = 1; jj <= P; ++jj, ++it) {
                const uint32_t buf = it & 1;
                const uint32_t buf_phase = (it >> 1) & 1;
                int got = lane == 0 ? (int)wait_bar(tfull_bar + 8 * buf, buf_phase, ab, 6) : 0;
                got = __shfl_sync(0xFFFFFFFFu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < BN / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + cc * 32, v);
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        const uint32_t c = pack_bf16x2(v[2 * w], v[2 * w + 1]);   // C_r = bf16(partial)
                        acc[cc * 16 + w] = jj == 1 ? c : add_bf16x2_bits(acc[cc * 16 + w], c);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar + 8 * buf);
            }
            if (!ok) break;
            const size_t row = (size_t)m * BM + q * 32 + lane;
            const size_t col = (size_t)n * BN - (size_t)k * p.n_chunk;   // column inside chunk k
            char *dst = p.out + (size_t)k * p.out_stride + (row * (size_t)p.n_chunk + col) * 2;
            if (p.st32) {
#pragma unroll
                for (int w = 0; w < BN / 16; ++w)   // one full 32-byte sector per lane and store
                    st8<OUT_POL>(dst + w * 32, make_uint4(acc[8 * w], acc[8 * w + 1], acc[8 * w + 2], acc[8 * w + 3]),
                                   make_uint4(acc[8 * w + 4], acc[8 * w + 5], acc[8 * w + 6], acc[8 * w + 7]));
            } else {
#pragma unroll
                for (int w = 0; w < BN / 8; ++w)
                    st_v4(dst + w * 16, make_uint4(acc[4 * w], acc[4 * w + 1], acc[4 * w + 2], acc[4 * w + 3]));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
}

// ------------------------------------------------------------ CTA-pair form
// The same computation on 256x256 output tiles, each run by a 2-CTA cluster:
// CTA c of the pair loads rows [128c, 128c+128) of the tile's A block and
// rows [128c, 128c+128) of its B block, and the even CTA issues
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16), which reads both CTAs'
// halves and leaves each CTA's 128 rows of D in its own TMEM.
// Operand staging is sized to the tile loader (TMA): measured on GB300, one
// SM's tiled loads top out near 70 bytes per clock.  A stage is K=128 deep by
// default (gemm_cfg.h) and each operand half arrives as one 32 KiB request (a
// box of two 64-column K blocks of 128 rows): 64 KiB per CTA per 1024 MMA
// clocks, under that ceiling, where the one-CTA 128x256 tile needs 94 bytes
// per clock.  With P=1 this kernel is a plain GEMM: 8192x4096x4096 bf16 runs
// in 0.154 ms on GB300, 91 % of cuBLAS on the same shape.
//   even CTA: warp 0 A producer (arms the stage's full barrier for the bytes
//             of both CTAs), warp 3 B producer, warp 1 MMA issuer, warps 4..
//             epilogue.
//   odd CTA:  warps 0 and 3 producers (their loads complete on the even CTA's
//             full barrier), warps 4.. epilogue (arrive on the even CTA's
//             accumulator-empty barrier).
// Both CTAs allocate TMEM together (.cta_group::2) and meet at cluster
// barriers after set-up and before freeing TMEM.
constexpr int PM = 256;                 // pair tile rows
constexpr int PN = 256;                 // pair tile columns
constexpr int HM = 128, HN = 128;       // per-CTA halves of A rows and B rows
constexpr int BK2 = RC_GEMM_PAIR_BK;    // K per stage: KSUB2 64-column swizzled sub-tiles
constexpr int KSUB2 = BK2 / 64;
constexpr int STAGES2 = RC_GEMM_PAIR_STAGES;
constexpr int A2_SUB = HM * 64 * 2;     // 16 KiB: one K sub-tile of the A half
constexpr int B2_SUB = HN * 64 * 2;
constexpr int A2_STAGE = KSUB2 * A2_SUB;
constexpr int B2_STAGE = KSUB2 * B2_SUB;
constexpr int SMEM2_BYTES = STAGES2 * (A2_STAGE + B2_STAGE) + 1024 + 256;
constexpr uint32_t kIdesc2 = idesc_bf16_f32(PM, PN);
// Epilogue warps of the pair kernel: 4 (one per TMEM lane quadrant, all 256
// columns each) or 8 (two per quadrant, 128 columns each).  Every partial
// product of a tile must be folded before the MMA warp needs its accumulator
// again, i.e. within the 32 K=16 MMAs of one partial (K=512 per rank).
// Measured on GB300 (P=8, 8192x4096x512 per rank): 4 warps 0.1779 ms,
// 8 warps 0.1776-0.1789 ms with the two-step hop add; 0.1698 vs 0.1697 ms
// with the one-instruction add (add_bf16x2_bits in dev.cuh).
#ifndef RC_GRS_EPI_WARPS
#define RC_GRS_EPI_WARPS 4
#endif
constexpr int EPI2 = RC_GRS_EPI_WARPS;
static_assert(EPI2 == 4 || EPI2 == 8, "one or two epilogue warps per TMEM lane quadrant");
constexpr int THREADS2 = 128 + 32 * EPI2;
constexpr int CW2 = PN / (EPI2 / 4);     // accumulator columns per epilogue warp
// 1: the last partial's fold stores each finished 32-column group at once
// (measured on GB300: 0.1757-0.1771 ms vs 0.1786-0.1788 ms storing the tile
// after the fold with the two-step hop add; 0.1698-0.1702 vs 0.1692 ms with
// the one-instruction add).
#ifndef RC_GRS_STORE_IN_FOLD
#define RC_GRS_STORE_IN_FOLD 1
#endif

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS2, 1)
    k_gemm_rs2(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = sA + STAGES2 * A2_STAGE;
    uint8_t *bars_g = gbase + STAGES2 * (A2_STAGE + B2_STAGE);
    const uint32_t bars = smem_u32(bars_g);
    const uint32_t full_bar = bars, empty_bar = bars + 8 * STAGES2;
    const uint32_t tfull_bar = bars + 16 * STAGES2, tempty_bar = tfull_bar + 16;
    const uint32_t drain_bar = tempty_bar + 16;
    uint32_t *tmem_slot = (uint32_t *)(bars_g + 16 * STAGES2 + 40);
    int *abort_flag = (int *)(bars_g + 16 * STAGES2 + 44);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t cta = cluster_ctarank();
    const bool even = cta == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(full_bar + 8 * s, 1);      // the even CTA's arm (expect_tx) is its one arrival
            mbar_init(empty_bar + 8 * s, 1);     // one commit of the pair's MMAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar + 8 * a, 1);
            mbar_init(tempty_bar + 8 * a, 2 * EPI2);   // every epilogue warp of both CTAs
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_b) : "memory");
    }
    // Both CTAs are running and their barriers initialised before the
    // collective TMEM allocation (one warp of each CTA) and any remote arrival.
    __syncthreads();
    cluster_sync_all();
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t full_even = mapa_shared(full_bar, 0);      // the even CTA's barriers
    const uint32_t tempty_even = mapa_shared(tempty_bar, 0);
    const Abort ab{abort_flag, p.hdr, p.timeout_ns, 0xA8u, mapa_shared(smem_u32(abort_flag), cta ^ 1u)};
    const int ksteps = p.K / BK2;
    const int P = p.P;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    // Producers: warp 0 loads the A halves (and, in the even CTA, arms the
    // full barrier for all four loads of the stage); with RC_GEMM_SPLIT_PRODUCER
    // warp 3 loads the B halves, so the two requests of a stage are in flight
    // together instead of one after the other.
    const bool a_producer = warp == 0 && lane == 0;
    const bool b_producer = (RC_GEMM_SPLIT_PRODUCER ? warp == 3 : warp == 0) && lane == 0;
    if (a_producer || b_producer) {
        // ---------------- TMA producer (both CTAs)
        uint32_t stage = 0, phase = 0;
        int issued[STAGES2] = {};
        bool ok = true;
        for (int t = pair; t < p.total_tiles && ok; t += npairs) {
            const int m = t / p.n_tiles, n = t % p.n_tiles;
            const int k = (n * PN) / p.n_chunk;
            for (int jj = 1; jj <= P && ok; ++jj) {
                const int r = (k + jj) % P;
                for (int kb = 0; kb < ksteps; ++kb) {
                    if (!wait_bar(empty_bar + 8 * stage, phase ^ 1u, ab, 2)) {
                        ok = false;
                        break;
                    }
                    if (a_producer) {
                        if (even) mbar_expect_tx(full_bar + 8 * stage, 2 * (A2_STAGE + B2_STAGE));
                        tma_load_4d_pair(sA + stage * A2_STAGE, &map_a, 0, m * PM + (int)cta * HM, kb * KSUB2, r,
                                         full_even + 8 * stage);
                    }
                    if (b_producer)
                        tma_load_4d_pair(sB + stage * B2_STAGE, &map_b, 0, n * PN + (int)cta * HN, kb * KSUB2, r,
                                         full_even + 8 * stage);
                    issued[stage]++;
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        // The even CTA's full barriers count both CTAs' bytes: once the last
        // phase armed on each has completed, no load of either CTA is in flight.
        if (a_producer && even && *(volatile int *)abort_flag) {
            for (int s = 0; s < STAGES2; ++s)
                if (issued[s] > 0) wait_bar(full_bar + 8 * s, (uint32_t)((issued[s] - 1) & 1), ab, 9, true);
        }
    } else if (warp == 1 && lane == 0 && even) {
        // ---------------- MMA issuer (even CTA)
        uint32_t stage = 0, phase = 0;
        int it = 0;
        bool ok = true;
        for (int t = pair; t < p.total_tiles && ok; t += npairs) {
            for (int jj = 1; jj <= P; ++jj, ++it) {
                const uint32_t acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!wait_bar<true>(tempty_bar + 8 * acc, acc_phase ^ 1u, ab, 3)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * PN;
                for (int kb = 0; kb < ksteps; ++kb) {
                    if (!wait_bar(full_bar + 8 * stage, phase, ab, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BK2 / UK; ++kk) {
                        // sub-tile kk/4 of the stage, then 32 bytes per K=16 step inside its swizzled rows
                        const uint64_t ad = smem_desc_sw128(sA + stage * A2_STAGE + (kk >> 2) * A2_SUB);
                        const uint64_t bd = smem_desc_sw128(sB + stage * B2_STAGE + (kk >> 2) * B2_SUB);
                        tc_mma_pair(d, ad + (uint64_t)(2 * (kk & 3)), bd + (uint64_t)(2 * (kk & 3)), kIdesc2,
                                    (kb | kk) != 0);
                    }
                    tc_commit_pair_mc(empty_bar + 8 * stage, 3);   // frees the stage in both CTAs
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit_pair_mc(tfull_bar + 8 * acc, 3);       // both CTAs' halves of D are ready
                if (!ok) break;
            }
        }
        tc_commit_pair_mc(drain_bar, 1);
        wait_bar(drain_bar, 0, ab, 10, true);
    } else if (warp >= 4) {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows of the pair tile.
        // Warp 4+e reads TMEM lane quadrant e % 4 (a warp may only access the
        // 32 lanes of its own warp index modulo 4) and columns [c0, c0 + CW2).
        const int e = warp - 4;
        const int q = e & 3;
        const int c0 = (e >> 2) * CW2;
        int it = 0;
        bool ok = true;
        for (int t = pair; t < p.total_tiles && ok; t += npairs) {
            const int m = t / p.n_tiles, n = t % p.n_tiles;
            const int k = (n * PN) / p.n_chunk;
            const size_t row = (size_t)m * PM + cta * HM + q * 32 + lane;
            const size_t col = (size_t)n * PN - (size_t)k * p.n_chunk + (size_t)c0;
            char *dst = p.out + (size_t)k * p.out_stride + (row * (size_t)p.n_chunk + col) * 2;
            uint32_t acc[CW2 / 2];
            for (int jj = 1; jj <= P; ++jj, ++it) {
                const uint32_t buf = it & 1;
                const uint32_t buf_phase = (it >> 1) & 1;
                int got = lane == 0 ? (int)wait_bar(tfull_bar + 8 * buf, buf_phase, ab, 6) : 0;
                got = __shfl_sync(0xFFFFFFFFu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Two 32-column loads in flight: the next is issued before this one is folded.
                // The last partial's fold stores each finished 32-column group at once
                // (RC_GRS_STORE_IN_FOLD), so the tile's stores overlap its TMEM loads.
                const bool last = RC_GRS_STORE_IN_FOLD && jj == P;
                const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + buf * PN + (uint32_t)c0;
                uint32_t va[32], vb[32];
                tmem_ld32_async(trow, va);
#pragma unroll
                for (int cc = 0; cc < CW2 / 32; cc += 2) {
                    tmem_wait_ld32(va);
                    tmem_ld32_async(trow + (cc + 1) * 32, vb);
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        const uint32_t c = pack_bf16x2(va[2 * w], va[2 * w + 1]);
                        acc[cc * 16 + w] = jj == 1 ? c : add_bf16x2_bits(acc[cc * 16 + w], c);
                    }
                    if (last && p.st32) {
#pragma unroll
                        for (int w = 0; w < 2; ++w)   // one full 32-byte sector per lane and store
                            st8<OUT_POL>(dst + cc * 64 + w * 32,
                                           make_uint4(acc[cc * 16 + 8 * w], acc[cc * 16 + 8 * w + 1],
                                                      acc[cc * 16 + 8 * w + 2], acc[cc * 16 + 8 * w + 3]),
                                           make_uint4(acc[cc * 16 + 8 * w + 4], acc[cc * 16 + 8 * w + 5],
                                                      acc[cc * 16 + 8 * w + 6], acc[cc * 16 + 8 * w + 7]));
                    } else if (last) {
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            st_v4(dst + cc * 64 + w * 16,
                                  make_uint4(acc[cc * 16 + 4 * w], acc[cc * 16 + 4 * w + 1],
                                             acc[cc * 16 + 4 * w + 2], acc[cc * 16 + 4 * w + 3]));
                    }
                    tmem_wait_ld32(vb);
                    if (cc + 2 < CW2 / 32) tmem_ld32_async(trow + (cc + 2) * 32, va);
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        const uint32_t c = pack_bf16x2(vb[2 * w], vb[2 * w + 1]);
                        acc[(cc + 1) * 16 + w] = jj == 1 ? c : add_bf16x2_bits(acc[(cc + 1) * 16 + w], c);
                    }
                    if (last && p.st32) {
#pragma unroll
                        for (int w = 0; w < 2; ++w)   // one full 32-byte sector per lane and store
                            st8<OUT_POL>(dst + (cc + 1) * 64 + w * 32,
                                           make_uint4(acc[(cc + 1) * 16 + 8 * w], acc[(cc + 1) * 16 + 8 * w + 1],
                                                      acc[(cc + 1) * 16 + 8 * w + 2], acc[(cc + 1) * 16 + 8 * w + 3]),
                                           make_uint4(acc[(cc + 1) * 16 + 8 * w + 4], acc[(cc + 1) * 16 + 8 * w + 5],
                                                      acc[(cc + 1) * 16 + 8 * w + 6], acc[(cc + 1) * 16 + 8 * w + 7]));
                    } else if (last) {
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            st_v4(dst + (cc + 1) * 64 + w * 16,
                                  make_uint4(acc[(cc + 1) * 16 + 4 * w], acc[(cc + 1) * 16 + 4 * w + 1],
                                             acc[(cc + 1) * 16 + 4 * w + 2], acc[(cc + 1) * 16 + 4 * w + 3]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (even)
                        mbar_arrive(tempty_bar + 8 * buf);
                    else
                        arrive_remote_relaxed(tempty_even + 8 * buf);
                }
            }
            if (!ok) break;
            if (!RC_GRS_STORE_IN_FOLD && p.st32) {
#pragma unroll
                for (int w = 0; w < CW2 / 16; ++w)
                    st8<OUT_POL>(dst + w * 32, make_uint4(acc[8 * w], acc[8 * w + 1], acc[8 * w + 2], acc[8 * w + 3]),
                                   make_uint4(acc[8 * w + 4], acc[8 * w + 5], acc[8 * w + 6], acc[8 * w + 7]));
            } else if (!RC_GRS_STORE_IN_FOLD) {
#pragma unroll
                for (int w = 0; w < CW2 / 8; ++w)
                    st_v4(dst + w * 16, make_uint4(acc[4 * w], acc[4 * w + 1], acc[4 * w + 2], acc[4 * w + 3]));
            }
        }
    }

    // Teardown: no MMA of the pair is in flight (the even CTA drained them) and
    // no epilogue still reads TMEM once both CTAs pass the cluster barrier.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

static int make_map3(CUtensorMap *map, const void *ptr, size_t K, size_t rows, int P, size_t rank_stride,
                     uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return set_error(RC_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)P};
    cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)rank_stride};
    cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(RC_ERR_INVALID, "tensor map encoding failed (CUresult %d)", (int)r);
    return RC_OK;
}

// Tuning knob, read once from the environment: RC_GEMM_PAIRS=0 keeps the
// one-CTA kernel even where the CTA-pair form applies (M a multiple of 256).
static bool pair_tiles_enabled()
{
    static const bool v = [] {
        const char *e = getenv("RC_GEMM_PAIRS");
        return !(e && e[0] == '0' && e[1] == 0);
    }();
    return v;
}

// The same operand as [P][K/64][rows][64]: a box of two 64-column K blocks of
// box_rows rows is one request (the CTA-pair kernel's 32 KiB stages).
static int make_map4(CUtensorMap *map, const void *ptr, size_t K, size_t rows, int P, size_t rank_stride,
                     uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return set_error(RC_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)K / 64, (cuuint64_t)P};
    cuuint64_t strides[3] = {(cuuint64_t)K * 2, 128, (cuuint64_t)rank_stride};
    cuuint32_t box[4] = {64, box_rows, (cuuint32_t)KSUB2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(RC_ERR_INVALID, "tensor map encoding failed (CUresult %d)", (int)r);
    return RC_OK;
}

static bool overlap(const void *a, size_t an, const void *b, size_t bn)
{
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bn && b0 < a0 + an;
}

} // namespace grs
} // namespace rc

static int gemm_rs_run(const void *A, size_t a_stride, const void *B, size_t b_stride, void *out, size_t out_stride,
                       int P, int M, int N, int K, void *ws, size_t ws_bytes, void *stream)
{
    using namespace rc;
    using namespace rc::grs;
    if (P < 1 || P > RC_MAX_P) return set_error(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (M <= 0 || N <= 0 || K <= 0 || M % BM || K % BK || N % P || (N / P) % BN)
        return set_error(RC_ERR_INVALID, "need M %% %d == 0, K %% %d == 0 and N/P a multiple of %d (got M=%d N=%d K=%d P=%d)",
                         BM, BK, BN, M, N, K, P);
    if (!A || !B || !out) return set_error(RC_ERR_INVALID, "null pointer");
    if (((uintptr_t)A | (uintptr_t)B | (uintptr_t)out | a_stride | b_stride | out_stride) & 15u)
        return set_error(RC_ERR_INVALID, "pointers and strides must be 16-byte aligned");
    const size_t a_bytes = (size_t)M * K * 2, b_bytes = (size_t)N * K * 2;
    const size_t n_chunk = (size_t)N / P, o_bytes = (size_t)M * n_chunk * 2;
    if (P > 1 && (a_stride < a_bytes || b_stride < b_bytes || out_stride < o_bytes))
        return set_error(RC_ERR_INVALID, "a stride is below the bytes of a rank's operand");
    const size_t a_span = (size_t)(P - 1) * a_stride + a_bytes, b_span = (size_t)(P - 1) * b_stride + b_bytes;
    const size_t o_span = (size_t)(P - 1) * out_stride + o_bytes;
    if (overlap(out, o_span, A, a_span) || overlap(out, o_span, B, b_span))
        return set_error(RC_ERR_INVALID, "out overlaps an input");

    Params p{};
    p.out = (char *)out;
    p.out_stride = P > 1 ? out_stride : o_bytes;
    p.P = P;
    p.M = M;
    p.N = N;
    p.K = K;
    p.n_chunk = (int)n_chunk;
    p.st32 = (((uintptr_t)out | p.out_stride | n_chunk * 2) & 31u) == 0;
    int sm_count = 0;
    uint32_t *unused = nullptr;
    int rc_ = prepare_workspace_ext(ws, ws_bytes, 0, &p.hdr, &unused, &sm_count, &p.timeout_ns);
    if (rc_) return rc_;
    const bool pairs = M % PM == 0 && K % BK2 == 0 && sm_count >= 2 && pair_tiles_enabled();
    CUtensorMap map_a, map_b;
    const size_t ars = P > 1 ? a_stride : a_bytes, brs = P > 1 ? b_stride : b_bytes;
    if (pairs) {
        if ((rc_ = make_map4(&map_a, A, (size_t)K, (size_t)M, P, ars, HM))) return rc_;
        if ((rc_ = make_map4(&map_b, B, (size_t)K, (size_t)N, P, brs, HN))) return rc_;
    } else {
        if ((rc_ = make_map3(&map_a, A, (size_t)K, (size_t)M, P, ars, BM))) return rc_;
        if ((rc_ = make_map3(&map_b, B, (size_t)K, (size_t)N, P, brs, BN))) return rc_;
    }
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(k_gemm_rs, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(k_gemm_rs2, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM2_BYTES);
    });
    if (attr_err != cudaSuccess)
        return set_error(RC_ERR_CUDA, "shared-memory attribute: %s", cudaGetErrorString(attr_err));
    if (pairs) {
        p.m_tiles = M / PM;
        p.n_tiles = N / PN;
        p.total_tiles = p.m_tiles * p.n_tiles;
        int clusters = sm_count / 2;
        if (clusters > p.total_tiles) clusters = p.total_tiles;
        k_gemm_rs2<<<2 * clusters, THREADS2, SMEM2_BYTES, (cudaStream_t)stream>>>(map_a, map_b, p);
    } else {
        p.m_tiles = M / BM;
        p.n_tiles = N / BN;
        p.total_tiles = p.m_tiles * p.n_tiles;
        int grid = sm_count;
        if (grid > p.total_tiles) grid = p.total_tiles;
        k_gemm_rs<<<grid, THREADS, SMEM_BYTES, (cudaStream_t)stream>>>(map_a, map_b, p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(RC_ERR_CUDA, "gemm_rs launch: %s", cudaGetErrorString(e));
    return RC_OK;
}

extern "C" int gemm_rs(const void *A, size_t a_stride, const void *B, size_t b_stride, void *out, size_t out_stride,
                       int P, int M, int N, int K, void *stream)
{
    return gemm_rs_run(A, a_stride, B, b_stride, out, out_stride, P, M, N, K, nullptr, 0, stream);
}

extern "C" int gemm_rs_ex(const void *A, size_t a_stride, const void *B, size_t b_stride, void *out,
                          size_t out_stride, int P, int M, int N, int K, void *workspace, size_t ws_bytes, void *stream)
{
    if (!workspace) return rc::set_error(RC_ERR_INVALID, "null workspace");
    return gemm_rs_run(A, a_stride, B, b_stride, out, out_stride, P, M, N, K, workspace, ws_bytes, stream);
}

// The launch keeps only its status header in the workspace.
extern "C" size_t gemm_rs_workspace_bytes(int P, int M, int N, int K)
{
    if (P < 1 || P > RC_MAX_P || M <= 0 || N <= 0 || K <= 0) return 0;
    return sizeof(rc::WsHeader);
}
