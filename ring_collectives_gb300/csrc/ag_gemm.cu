// ag_gemm.cu -- all-gather of row shards fused with C = A_g . B^T on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// Sources: "TPU 与分布式通信原语", section "collective matmul" (all-gather the
// row shards, then the local matmul with a bf16 result); "Triton-distributed
// 语义", sections "生产者-消费者模型" and "AllGather + GEMM 重叠" (a producer
// copies tiles and signals each one, a consumer waits per tile and computes
// at once) and "线程块交织" (pid_m = (pid_m + rank*tiles_per_pe) % total so
// every rank starts on its own, already local, rows).
//
// One persistent cooperative launch, one 256-thread block per SM:
//   warp 0      TMA producer: A and B tiles (128x64 and 256x64 bf16, 128-byte
//               swizzle) into a 4-stage shared-memory ring.  Before the first
//               A tile of an M block that came from another rank it needs
//               that block's ready flags set: it looks at them from half-way
//               through the previous tile on and, if it has not seen them by
//               the tile boundary, waits there (acquire, bounded).
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=256,
//               K=16, bf16 x bf16 -> fp32) into one of two TMEM accumulators
//               and releases smem stages / accumulators with tcgen05.commit.
//   warp 2      allocates TMEM (512 columns) and, on one thread, runs the
//               gather producer: 16-row pieces of the shards are copied into
//               A_g with bulk copies through 32 KiB of staging buffers, in
//               the order the consumers need them, and each piece publishes
//               its ready flag (st.release of the launch epoch); see
//               gather_units.  (The CTA-pair form below gathers on part of
//               the grid only.)
//   warps 4-7   epilogue: TMEM -> registers (tcgen05.ld), fp32 -> bf16 (RNE),
//               stores to C (evict_first), then free the accumulator for
//               the MMA warp.
// Rows of the own rank are read straight from its shard (local data, no
// wait); rows of other ranks come from A_g once their flags are set.
//
// Every wait (mbarrier or flag) is bounded by %globaltimer; a wait that runs
// out records RC_ERR_TIMEOUT in the workspace header and makes every role of
// the block stop; in-flight copies and MMAs are drained (also bounded) and
// TMEM is freed before the block exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "gemm_cfg.h"
#include "tc.cuh"

namespace rc {
namespace ag {

constexpr int BM = 128, BN = 256, BK = 64, UK = 16;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;   // 16 KiB
constexpr int B_STAGE = BN * BK * 2;   // 32 KiB
// Gather staging buffer bytes (two of them).  Measured on GB300 (P=8,
// 8192x4096x4096, one box): 4 KiB 0.177 ms, 8 KiB 0.171, 16 KiB 0.169;
// larger does not fit beside three 64 KiB operand stages.
#ifndef RC_AG_GEMM_STAGING
#define RC_AG_GEMM_STAGING 16384
#endif
constexpr int STAGING = RC_AG_GEMM_STAGING; // gather staging buffer (x2)
// The A producer looks at the ready flags of its next tile
// half-way through the current one and then every RC_AG_POLL_EVERY stages
// until it sees them set (0: only the one look half-way through).
#ifndef RC_AG_POLL_EVERY
#define RC_AG_POLL_EVERY 4
#endif
constexpr int POLL_EVERY = RC_AG_POLL_EVERY > 0 ? RC_AG_POLL_EVERY : 1 << 20;
// Gather copies with L2 eviction hints (1): other ranks' shard rows, read
// once, are loaded evict_first so that they do not push the GEMM's operands
// out of L2.
#ifndef RC_AG_GATHER_HINT
#define RC_AG_GATHER_HINT 1
#endif
// The gather's staging space (2 x STAGING bytes) as a ring of
// RC_AG_GATHER_BUFS buffers, all but one of them loading at any time.
#ifndef RC_AG_GATHER_BUFS
#define RC_AG_GATHER_BUFS 4
#endif
constexpr int GB = RC_AG_GATHER_BUFS;
// C, which nothing reads in the launch, is stored
// evict_first (RC_AG_C_POLICY 1; 0 normal), so that the 64 MiB it streams
// through L2 does not push out operand rows still to be read.
#ifndef RC_AG_C_POLICY
#define RC_AG_C_POLICY 1
#endif
constexpr int C_POL = RC_AG_C_POLICY ? kStEvictFirst : kStNormal;
// CTA-pair form, who gathers.  When the tiles do not divide evenly, pairs
// numbered below total_tiles % npairs run one tile more than the rest.  Per
// round of gather units, each CTA of such a pair takes RC_AG_GATHER_NW units
// and each CTA of the other pairs RC_AG_GATHER_SW: the gather's bulk copies
// share the SM's copy engine with the GEMM's operand loads, so they go where
// the SM has time to spare.
#ifndef RC_AG_GATHER_NW
#define RC_AG_GATHER_NW 0
#endif
#ifndef RC_AG_GATHER_SW
#define RC_AG_GATHER_SW 1
#endif
static_assert(RC_AG_GATHER_NW >= 0 && RC_AG_GATHER_SW >= 1, "every round needs a gathering CTA");
constexpr int GCH = 2 * STAGING / GB;   // bytes per gather buffer
static_assert(GB >= 2 && GB <= 8 && GCH % 16 == 0, "gather ring: 2..8 buffers of whole 16-byte units");
constexpr int PIECE_ROWS = 16;         // rows per gather unit (one ready flag each)
constexpr int THREADS = 256;
constexpr int TMEM_COLS = 512;         // two 128x256 fp32 accumulators
constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) + 2 * STAGING + 1024 /*align*/ + 256 /*barriers*/;

struct Params {
    const char *a_shards;
    size_t a_stride;
    char *a_gathered;
    char *C;
    uint32_t *flags;     // one per gather unit
    WsHeader *hdr;
    int P, rank, M_r, N, K;
    int total_m, tiles_per_pe, n_tiles, total_tiles, units;  // tile schedule (tile rows: BM, or PM for pairs)
    int g_total_m, g_per_pe;   // gather schedule, in 128-row blocks (8 units of 16 rows each)
    int st32;                  // 1: rows of C start on 32-byte boundaries (full-sector stores)
    int b_kn;                  // 1: B is stored [K][N] (MN-major operand), 0: [N][K] (K-major)
    int skip_row;              // test hook: the piece starting at this A_g row is never published (-1: none)
    unsigned long long timeout_ns;
};

// ------------------------------------------------------------ PTX wrappers (tc.cuh)
using namespace tc;
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

// Stores the 32 columns of one TMEM load (fp32, rounded to bf16) of this
// lane's row of C.  Each lane owns a row, so a warp's store touches 32 rows;
// 32-byte stores fill whole sectors (measured on GB300: the 16-byte form
// costs the epilogue about twice the store time).
template <int POL = kStNormal>
__device__ __forceinline__ void store_row32(char *dst, const uint32_t (&v)[32], bool st32)
{
    uint32_t b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) b[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    if (st32) {
        st8<POL>(dst, make_uint4(b[0], b[1], b[2], b[3]), make_uint4(b[4], b[5], b[6], b[7]));
        st8<POL>(dst + 32, make_uint4(b[8], b[9], b[10], b[11]), make_uint4(b[12], b[13], b[14], b[15]));
    } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) st_v4(dst + w * 16, make_uint4(b[4 * w], b[4 * w + 1], b[4 * w + 2], b[4 * w + 3]));
    }
}

// ------------------------------------------------------------ tile order
// Tile t of the persistent schedule -> (m block, n block).  Raw M order is
// swizzled by rank so that the first M blocks are the rank's own rows.
__device__ __forceinline__ void tile_of(const Params &p, int t, int &m, int &n)
{
    const int m_raw = t / p.n_tiles;
    n = t % p.n_tiles;
    m = (m_raw + p.rank * p.tiles_per_pe) % p.total_m;
}

// Gather unit u (in the order the consumers need them: other ranks' M blocks
// in swizzled order, the own rank's last) -> (M block, piece).
__device__ __forceinline__ void unit_of(const Params &p, int u, int &mb, int &piece)
{
    const int pieces = BM / PIECE_ROWS;
    const int i = u / pieces;
    piece = u % pieces;
    const int others = p.g_total_m - p.g_per_pe;
    const int order = i < others ? i + p.g_per_pe : i - others;
    mb = (order + p.rank * p.g_per_pe) % p.g_total_m;
}

// Waits until the BM/PIECE_ROWS ready flags of one 128-row block of A_g have
// reached the launch's epoch.  The flags are read together (relaxed loads,
// one round trip per poll instead of one per flag); the fence.acq_rel after
// the poll that saw them all makes those reads an acquire, so with the gather
// producers' release stores every copy into the block precedes what follows.
// Bounded like every other wait.
__device__ bool wait_block_flags(const uint32_t *f, uint32_t E, const Abort &ab, int where)
{
    constexpr int NF = BM / PIECE_ROWS;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t v[NF];
#pragma unroll
        for (int q = 0; q < NF; ++q) v[q] = ld_relaxed_gpu(f + q);
        bool all = true;
#pragma unroll
        for (int q = 0; q < NF; ++q) all = all && epoch_reached(v[q], E);
        if (all) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            return true;
        }
        if ((it & 15u) == 15u) {
            if (*(volatile int *)ab.flag) return false;
            const uint64_t now = global_timer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > ab.timeout_ns) {
                record_timeout(ab, where);
                return false;
            }
        }
        __nanosleep(64);
    }
}

// One non-blocking look at the ready flags of a 128-row block of A_g: true
// (after an acquire fence, as in wait_block_flags) if all of them have
// reached the launch's epoch.
__device__ bool poll_block_flags(const uint32_t *f, uint32_t E)
{
    constexpr int NF = BM / PIECE_ROWS;
    uint32_t v[NF];
#pragma unroll
    for (int q = 0; q < NF; ++q) v[q] = ld_relaxed_gpu(f + q);
    bool all = true;
#pragma unroll
    for (int q = 0; q < NF; ++q) all = all && epoch_reached(v[q], E);
    if (all) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    return all;
}

// Gather producer (one thread per CTA): copies gather units into A_g and
// publishes each unit's ready flag (st.release of the launch epoch).  This
// CTA takes units first, first+1, ..., first+w-1, then the same w units
// per_round further on, and so on.  Each unit (PIECE_ROWS rows) streams
// through a ring of GB staging buffers at sStage with barriers at gat_bar: a
// load (global -> shared) per buffer in flight, and a buffer refilled once
// the store (shared -> A_g) of its previous chunk has read it.  Other
// ranks' rows, read once here, are loaded evict_first.  Bounded waits; on
// a failure every load still in flight lands before the function returns.
__device__ void gather_units(const Params &p, uint32_t sStage, uint32_t gat_bar, const Abort &ab,
                             const int *abort_flag, uint32_t E, int first, int per_round, int w)
{
    const size_t row_bytes = (size_t)p.K * 2;
    const size_t unit_bytes = (size_t)PIECE_ROWS * row_bytes;
    const int nch = (int)((unit_bytes + GCH - 1) / GCH);
    const uint64_t pol_once = policy_evict_first();
    uint32_t gph = 0;   // bit b: parity of gather buffer b's next completion
    for (int i = 0; w > 0 && !*(volatile const int *)abort_flag; ++i) {
        const int u = first + (i / w) * per_round + i % w;   // increasing in i
        if (u >= p.units) break;
        int mb, piece;
        unit_of(p, u, mb, piece);
        const int row = mb * BM + piece * PIECE_ROWS;     // row of A_g
        const int src_rank = row / p.M_r;
        const char *src = p.a_shards + (size_t)src_rank * p.a_stride + (size_t)(row % p.M_r) * row_bytes;
        char *dst = p.a_gathered + (size_t)row * row_bytes;
        // Other ranks' rows are read once here (the GEMM reads them from
        // A_g); the own rank's rows are also the GEMM's operand.
        const bool once = RC_AG_GATHER_HINT && src_rank != p.rank;
        auto chunk_bytes = [&](int c) -> uint32_t {
            const size_t off = (size_t)c * GCH;
            return (uint32_t)(unit_bytes - off < (size_t)GCH ? unit_bytes - off : (size_t)GCH);
        };
        auto load = [&](int c) {
            const int b = c % GB;
            mbar_expect_tx(gat_bar + 8 * b, chunk_bytes(c));
            if (once)
                bulk_g2s_hint(sStage + b * GCH, src + (size_t)c * GCH, chunk_bytes(c), gat_bar + 8 * b, pol_once);
            else
                bulk_g2s(sStage + b * GCH, src + (size_t)c * GCH, chunk_bytes(c), gat_bar + 8 * b);
        };
        int issued = 0;
        for (; issued < nch && issued < GB; ++issued) load(issued);
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int b = c % GB;
            if (!wait_bar(gat_bar + 8 * b, (gph >> b) & 1u, ab, 5)) {
                // leave no load in flight: chunks c .. issued-1, one per buffer
                for (int d = c; d < issued; ++d) {
                    const int bd = d % GB;
                    wait_bar(gat_bar + 8 * bd, (gph >> bd) & 1u, ab, 11, true);
                    gph ^= 1u << bd;
                }
                ok = false;
                break;
            }
            gph ^= 1u << b;
            bulk_s2g(dst + (size_t)c * GCH, sStage + b * GCH, chunk_bytes(c));
            bulk_commit();
            if (c >= 1 && issued < nch) {   // chunk c-1's buffer, once its store has read it
                bulk_wait_read1();
                load(issued++);
            }
        }
        bulk_wait_all();              // this unit's rows are in A_g
        if (!ok) break;
        fence_proxy_async_global();   // async-proxy writes before the generic release
        if (row != p.skip_row) st_release_gpu(&p.flags[mb * (BM / PIECE_ROWS) + piece], E);
    }
    bulk_wait_all();
}

__global__ void __launch_bounds__(THREADS, 1)
    k_ag_gemm(const __grid_constant__ CUtensorMap map_ag, const __grid_constant__ CUtensorMap map_sh,
              const __grid_constant__ CUtensorMap map_b, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128-byte swizzle wants 1024-byte aligned tiles
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = sA + STAGES * A_STAGE;
    const uint32_t sStage = sB + STAGES * B_STAGE;
    uint8_t *bars_g = gbase + STAGES * (A_STAGE + B_STAGE) + 2 * STAGING;
    const uint32_t bars = smem_u32(bars_g);
    const uint32_t full_bar = bars, empty_bar = bars + 8 * STAGES;
    const uint32_t tfull_bar = bars + 16 * STAGES, tempty_bar = tfull_bar + 16;
    const uint32_t gat_bar = tempty_bar + 16;          // GB gather buffers
    const uint32_t drain_bar = gat_bar + 8 * GB;
    uint32_t *tmem_slot = (uint32_t *)(bars_g + 16 * STAGES + 40 + 8 * GB);
    int *abort_flag = (int *)(bars_g + 16 * STAGES + 44 + 8 * GB);
    uint32_t *epoch_slot = (uint32_t *)(bars_g + 16 * STAGES + 48 + 8 * GB);

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
        for (int b = 0; b < GB; ++b) mbar_init(gat_bar + 8 * b, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *epoch_slot = ld_relaxed_gpu(&p.hdr->epoch) + 1u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_ag) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_sh) : "memory");
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
    const uint32_t E = *epoch_slot;
    const Abort ab{abort_flag, p.hdr, p.timeout_ns, 0xA6u};
    const int ksteps = p.K / BK;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        uint32_t stage = 0, phase = 0;
        int issued[STAGES] = {0, 0, 0, 0};
        bool next_ready = false;   // the next tile's flags were already seen set (and acquired)
        for (int t = blockIdx.x; t < p.total_tiles && !*(volatile int *)abort_flag; t += gridDim.x) {
            int m, n;
            tile_of(p, t, m, n);
            const int src_rank = (m * BM) / p.M_r;
            const bool own = src_rank == p.rank;
            if (!own) {
                if (!next_ready && !wait_block_flags(&p.flags[m * (BM / PIECE_ROWS)], E, ab, 1)) break;
                fence_proxy_async_global(); // the generic-proxy flags order the async-proxy reads below
            }
            // the next tile's flags, looked at from half-way through this tile (as in the pair form)
            next_ready = false;
            const uint32_t *next_flags = nullptr;
            if (t + (int)gridDim.x < p.total_tiles) {
                int mn, nn;
                tile_of(p, t + (int)gridDim.x, mn, nn);
                if ((mn * BM) / p.M_r != p.rank) next_flags = &p.flags[mn * (BM / PIECE_ROWS)];
            }
            const int row_in_shard = (m * BM) % p.M_r;
            bool ok = true;
            for (int kb = 0; kb < ksteps; ++kb) {
                if (!wait_bar(empty_bar + 8 * stage, phase ^ 1u, ab, 2)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(full_bar + 8 * stage, A_STAGE + B_STAGE);
                if (own)
                    tma_load_3d(sA + stage * A_STAGE, &map_sh, kb * BK, row_in_shard, src_rank, full_bar + 8 * stage);
                else
                    tma_load_2d(sA + stage * A_STAGE, &map_ag, kb * BK, m * BM, full_bar + 8 * stage);
                if (p.b_kn)   // [K][N]: 4 blocks of 64 columns x BK rows of k
                    tma_load_3d(sB + stage * B_STAGE, &map_b, 0, kb * BK, n * (BN / 64), full_bar + 8 * stage);
                else
                    tma_load_2d(sB + stage * B_STAGE, &map_b, kb * BK, n * BN, full_bar + 8 * stage);
                issued[stage]++;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (next_flags && !next_ready && kb >= ksteps / 2 && (kb - ksteps / 2) % POLL_EVERY == 0)
                    next_ready = poll_block_flags(next_flags, E);
            }
            if (!ok) break;
        }
        // Drain: every load issued must have landed before the block may exit
        // (the last load into stage s completes phase (issued[s]-1) of full_bar[s]).
        if (*(volatile int *)abort_flag) {
            for (int s = 0; s < STAGES; ++s)
                if (issued[s] > 0) wait_bar(full_bar + 8 * s, (uint32_t)((issued[s] - 1) & 1), ab, 9, true);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        uint32_t stage = 0, phase = 0;
        int it = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
            const uint32_t acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            if (!wait_bar(tempty_bar + 8 * acc, acc_phase ^ 1u, ab, 3)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + acc * BN;
            bool ok = true;
            for (int kb = 0; kb < ksteps; ++kb) {
                if (!wait_bar(full_bar + 8 * stage, phase, ab, 4)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = smem_desc_sw128(sA + stage * A_STAGE);
                const uint64_t bd = p.b_kn ? smem_desc_mn_sw128(sB + stage * B_STAGE, BK * 128)
                                           : smem_desc_sw128(sB + stage * B_STAGE);
#pragma unroll
                for (int k = 0; k < BK / UK; ++k) {
                    // K advances 16 bf16 = 32 bytes inside the 128-byte swizzle row: +2 in 16-byte units;
                    // for an MN-major B it advances 16 rows of 128 bytes: +128
                    tc_mma(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(p.b_kn ? 128 * k : 2 * k),
                           kIdesc | (p.b_kn ? kIdescBMnMajor : 0u), (kb | k) != 0);
                }
                tc_commit(empty_bar + 8 * stage); // frees the smem stage once these MMAs have read it
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            tc_commit(tfull_bar + 8 * acc);       // accumulator ready once every MMA above completes
            if (!ok) break;
        }
        // Drain: no MMA may still read shared memory or write TMEM when the
        // block frees them; a commit after the last MMA tracks all of them.
        tc_commit(drain_bar);
        wait_bar(drain_bar, 0, ab, 10, true);
    } else if (warp == 2 && lane == 0) {
        // ---------------- gather producer (every CTA alike)
        gather_units(p, sStage, gat_bar, ab, abort_flag, E, (int)blockIdx.x, (int)gridDim.x, 1);
    } else if (warp >= 4) {
        // ---------------- epilogue
        const int q = warp - 4;            // TMEM lane quadrant of this warp
        int it = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
            const uint32_t acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            // One lane waits and the warp follows its result, so the warp stays
            // converged for the .sync.aligned TMEM loads below.
            int ok = lane == 0 ? (int)wait_bar(tfull_bar + 8 * acc, acc_phase, ab, 6) : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            int m, n;
            tile_of(p, t, m, n);
            const size_t row = (size_t)m * BM + q * 32 + lane;
            char *crow = p.C + row * (size_t)p.N * 2 + (size_t)n * BN * 2;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + cc * 32, v);
                store_row32<C_POL>(crow + cc * 64, v, p.st32);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar + 8 * acc);
        }
    }

    // ---------------- teardown (every role has drained its own async work)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&p.hdr->done, 1u);
        if (prev == gridDim.x - 1) {
            p.hdr->done = 0;
            st_relaxed_gpu(&p.hdr->epoch, E);
        }
    }
}

// ------------------------------------------------------------ CTA-pair form
// 256x256 tiles on 2-CTA clusters (the pair scheme of gemm_rs.cu): CTA c
// stages rows [128c, 128c+128) of the tile's A block and of its B block in
// K=128 stages (one 32 KiB box per operand half and stage, under the ~70
// bytes per clock per SM that tiled TMA loads reach on GB300), the even CTA
// issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and both CTAs drain
// their own 128 rows of D.  Each CTA waits only on the ready flags of its own
// 128 A rows.  Measured on GB300 (P=8, 8192x4096x4096, CUDA events over 30
// back-to-back calls), in both forms:
//  * the A producer looks at the next tile's flags from half-way through the
//    current tile (a flag round trip at the tile boundary left the MMA idle:
//    0.1633 -> 0.1604 ms);
//  * the gather streams each unit through a ring of 4 staging buffers with 3
//    loads in flight (one load at a time ran at ~10 GB/s per CTA), loading
//    other ranks' rows evict_first;
//  * C is stored evict_first (0.1592 -> 0.1552 ms).
// And in the pair form only:
//  * the gather runs on the CTAs of the pairs with one tile fewer: its bulk
//    copies share the SM's copy engine with the operand loads, and on the
//    pairs that set the launch's length it slowed the first tiles by ~3 us
//    each (0.1591 ms with every CTA gathering, 0.1580 with a 1:3 share,
//    0.1551 with the spare pairs alone).
// Without the gather and its waits the same kernel takes 0.1433 ms, as much
// as cuBLAS on the plain GEMM; in-kernel clock stamps put the SM clock at
// 1.6-1.9 GHz during the launch (the power limit), so tiles after the first
// run at ~94 % of the tensor pipe's per-cycle peak.
constexpr int PM = 256, PN = 256, HM = 128, HN = 128;
constexpr int BK2 = RC_GEMM_PAIR_BK;     // K per stage: KSUB2 64-column swizzled sub-tiles
constexpr int KSUB2 = BK2 / 64;
constexpr int STAGES2 = RC_GEMM_PAIR_STAGES;
constexpr int A2_SUB = HM * 64 * 2, B2_SUB = HN * 64 * 2;   // 16 KiB K sub-tiles
constexpr int A2_STAGE = KSUB2 * A2_SUB, B2_STAGE = KSUB2 * B2_SUB;
constexpr int SMEM2_BYTES = STAGES2 * (A2_STAGE + B2_STAGE) + 2 * STAGING + 1024 + 256;
constexpr uint32_t kIdesc2 = idesc_bf16_f32(PM, PN);

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k_ag_gemm2(const __grid_constant__ CUtensorMap map_ag, const __grid_constant__ CUtensorMap map_sh,
               const __grid_constant__ CUtensorMap map_b, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = sA + STAGES2 * A2_STAGE;
    const uint32_t sStage = sB + STAGES2 * B2_STAGE;
    uint8_t *bars_g = gbase + STAGES2 * (A2_STAGE + B2_STAGE) + 2 * STAGING;
    const uint32_t bars = smem_u32(bars_g);
    const uint32_t full_bar = bars, empty_bar = bars + 8 * STAGES2;
    const uint32_t tfull_bar = bars + 16 * STAGES2, tempty_bar = tfull_bar + 16;
    const uint32_t gat_bar = tempty_bar + 16;          // GB gather buffers
    const uint32_t drain_bar = gat_bar + 8 * GB;
    uint32_t *tmem_slot = (uint32_t *)(bars_g + 16 * STAGES2 + 40 + 8 * GB);
    int *abort_flag = (int *)(bars_g + 16 * STAGES2 + 44 + 8 * GB);
    uint32_t *epoch_slot = (uint32_t *)(bars_g + 16 * STAGES2 + 48 + 8 * GB);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t cta = cluster_ctarank();
    const bool even = cta == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar + 8 * a, 1);
            mbar_init(tempty_bar + 8 * a, 8);   // four epilogue warps of each CTA
        }
        for (int b = 0; b < GB; ++b) mbar_init(gat_bar + 8 * b, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *epoch_slot = ld_relaxed_gpu(&p.hdr->epoch) + 1u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_ag) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_sh) : "memory");
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
    const uint32_t E = *epoch_slot;
    const uint32_t full_even = mapa_shared(full_bar, 0);
    const uint32_t tempty_even = mapa_shared(tempty_bar, 0);
    const Abort ab{abort_flag, p.hdr, p.timeout_ns, 0xA9u, mapa_shared(smem_u32(abort_flag), cta ^ 1u)};
    const int ksteps = p.K / BK2;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    // Producers: warp 0 loads the A halves (and, in the even CTA, arms the
    // full barrier for all four loads of the stage); with RC_GEMM_SPLIT_PRODUCER
    // warp 3 loads the B halves, so the two requests of a stage are in flight
    // together instead of one after the other.
    const bool a_producer = warp == 0 && lane == 0;
    const bool b_producer = (RC_GEMM_SPLIT_PRODUCER ? warp == 3 : warp == 0) && lane == 0;
    if (a_producer || b_producer) {
        // ---------------- TMA producer (both CTAs): this CTA's halves of A and B
        uint32_t stage = 0, phase = 0;
        int issued[STAGES2] = {};
        bool next_ready = false;   // the next tile's flags were already seen set (and acquired)
        for (int t = pair; t < p.total_tiles && !*(volatile int *)abort_flag; t += npairs) {
            int m, n;
            tile_of(p, t, m, n);
            const int row0 = m * PM + (int)cta * HM;          // this CTA's 128 rows of A_g
            const int src_rank = row0 / p.M_r;
            const bool own = src_rank == p.rank;
            if (!own && a_producer) {
                if (!next_ready && !wait_block_flags(&p.flags[(row0 / BM) * (BM / PIECE_ROWS)], E, ab, 1)) break;
                fence_proxy_async_global();
            }
            // Looks at the next tile's flags: at the boundary the MMA has
            // only the last STAGES2 stages of this tile queued, less work than
            // one flag round trip plus one load; from half-way through the
            // tile on, each round trip hides behind the queued stages.  If no
            // look sees them set, the wait stays at the boundary.
            next_ready = false;
            const uint32_t *next_flags = nullptr;
            if (a_producer && t + npairs < p.total_tiles) {
                int mn, nn;
                tile_of(p, t + npairs, mn, nn);
                const int nrow0 = mn * PM + (int)cta * HM;
                if (nrow0 / p.M_r != p.rank) next_flags = &p.flags[(nrow0 / BM) * (BM / PIECE_ROWS)];
            }
            const int row_in_shard = row0 % p.M_r;
            bool ok = true;
            for (int kb = 0; kb < ksteps; ++kb) {
                if (!wait_bar(empty_bar + 8 * stage, phase ^ 1u, ab, 2)) {
                    ok = false;
                    break;
                }
                if (a_producer) {
                    if (even) mbar_expect_tx(full_bar + 8 * stage, 2 * (A2_STAGE + B2_STAGE));
                    if (own)
                        tma_load_4d_pair(sA + stage * A2_STAGE, &map_sh, 0, row_in_shard, kb * KSUB2, src_rank,
                                         full_even + 8 * stage);
                    else
                        tma_load_3d_pair(sA + stage * A2_STAGE, &map_ag, 0, row0, kb * KSUB2, full_even + 8 * stage);
                }
                if (b_producer) {
                    if (p.b_kn)   // [K][N]: this CTA's 2 blocks of 64 columns x BK2 rows of k
                        tma_load_3d_pair(sB + stage * B2_STAGE, &map_b, 0, kb * BK2, (n * PN + (int)cta * HN) / 64,
                                         full_even + 8 * stage);
                    else
                        tma_load_3d_pair(sB + stage * B2_STAGE, &map_b, 0, n * PN + (int)cta * HN, kb * KSUB2,
                                         full_even + 8 * stage);
                }
                issued[stage]++;
                if (++stage == STAGES2) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (next_flags && !next_ready && kb >= ksteps / 2 && (kb - ksteps / 2) % POLL_EVERY == 0)
                    next_ready = poll_block_flags(next_flags, E);
            }
            if (!ok) break;
        }
        // The even CTA's full barriers count both CTAs' bytes.
        if (a_producer && even && *(volatile int *)abort_flag) {
            for (int s = 0; s < STAGES2; ++s)
                if (issued[s] > 0) wait_bar(full_bar + 8 * s, (uint32_t)((issued[s] - 1) & 1), ab, 9, true);
        }
    } else if (warp == 1 && lane == 0 && even) {
        // ---------------- MMA issuer (even CTA)
        uint32_t stage = 0, phase = 0;
        int it = 0;
        for (int t = pair; t < p.total_tiles; t += npairs, ++it) {
            const uint32_t acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            if (!wait_bar<true>(tempty_bar + 8 * acc, acc_phase ^ 1u, ab, 3)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + acc * PN;
            bool ok = true;
            for (int kb = 0; kb < ksteps; ++kb) {
                if (!wait_bar(full_bar + 8 * stage, phase, ab, 4)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t bd_mn = smem_desc_mn_sw128(sB + stage * B2_STAGE, BK2 * 128);
#pragma unroll
                for (int kk = 0; kk < BK2 / UK; ++kk) {
                    const uint64_t ad = smem_desc_sw128(sA + stage * A2_STAGE + (kk >> 2) * A2_SUB);
                    // K-major B: 16 K-columns of a 64-column sub-tile; MN-major B: 16 rows of k (2048 bytes)
                    const uint64_t bd = p.b_kn ? bd_mn + (uint64_t)(128 * kk)
                                               : smem_desc_sw128(sB + stage * B2_STAGE + (kk >> 2) * B2_SUB) +
                                                     (uint64_t)(2 * (kk & 3));
                    tc_mma_pair(d, ad + (uint64_t)(2 * (kk & 3)), bd, kIdesc2 | (p.b_kn ? kIdescBMnMajor : 0u),
                                (kb | kk) != 0);
                }
                tc_commit_pair_mc(empty_bar + 8 * stage, 3);
                if (++stage == STAGES2) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            tc_commit_pair_mc(tfull_bar + 8 * acc, 3);
            if (!ok) break;
        }
        tc_commit_pair_mc(drain_bar, 1);
        wait_bar(drain_bar, 0, ab, 10, true);
    } else if (warp == 2 && lane == 0) {
        // ---------------- gather producer (units shared out by RC_AG_GATHER_NW / _SW)
        // The shares apply when the pairs with one tile fewer hold at least a
        // fifth of the grid: fewer CTAs could not copy the units as fast as
        // the consumers read them (one unit per CTA every ~6-8 us against
        // ~76 per 20 us wave at P=8, 8192x4096x4096), so then every CTA
        // gathers alike.
        const int full_pairs = p.total_tiles % npairs;
        const bool shares = full_pairs > 0 && 5 * 2 * (npairs - full_pairs) >= (int)gridDim.x;
        const int nw = shares ? RC_AG_GATHER_NW : 1, sw = shares ? RC_AG_GATHER_SW : 1;
        const int n_full = 2 * full_pairs;                                // CTAs of the pairs with the extra tile
        const int per_round = n_full * nw + ((int)gridDim.x - n_full) * sw;
        const bool spare = (int)blockIdx.x >= n_full;
        const int first = spare ? n_full * nw + ((int)blockIdx.x - n_full) * sw : (int)blockIdx.x * nw;
        gather_units(p, sStage, gat_bar, ab, abort_flag, E, first, per_round, spare ? sw : nw);
    } else if (warp >= 4) {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows of the pair tile
        const int q = warp - 4;
        int it = 0;
        for (int t = pair; t < p.total_tiles; t += npairs, ++it) {
            const uint32_t acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            int ok = lane == 0 ? (int)wait_bar(tfull_bar + 8 * acc, acc_phase, ab, 6) : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            int m, n;
            tile_of(p, t, m, n);
            const size_t row = (size_t)m * PM + cta * HM + q * 32 + lane;
            char *crow = p.C + row * (size_t)p.N * 2 + (size_t)n * PN * 2;
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + acc * PN;
            uint32_t va[32], vb[32];
            tmem_ld32_async(trow, va);
#pragma unroll
            for (int cc = 0; cc < PN / 32; cc += 2) {
                tmem_wait_ld32(va);
                tmem_ld32_async(trow + (cc + 1) * 32, vb);
                store_row32<C_POL>(crow + cc * 64, va, p.st32);
                tmem_wait_ld32(vb);
                if (cc + 2 < PN / 32) tmem_ld32_async(trow + (cc + 2) * 32, va);
                store_row32<C_POL>(crow + (cc + 1) * 64, vb, p.st32);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (even)
                    mbar_arrive(tempty_bar + 8 * acc);
                else
                    mbar_arrive_remote(tempty_even + 8 * acc);
            }
        }
    }

    // ---------------- teardown: no MMA of the pair in flight and no TMEM
    // reader left once both CTAs pass the cluster barrier.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&p.hdr->done, 1u);
        if (prev == gridDim.x - 1) {
            p.hdr->done = 0;
            st_relaxed_gpu(&p.hdr->epoch, E);
        }
    }
}

// ------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

// bf16 tensor map over `rank` dims (dims[0] innermost, strides in bytes for dims 1..),
// box {BK, box_rows, 1...}, 128-byte swizzle.
static int make_map(CUtensorMap *map, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return set_error(RC_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(RC_ERR_INVALID, "tensor map encoding failed (CUresult %d)", (int)r);
    return RC_OK;
}

// The same over [..][K/64][rows][64] (dims {64, rows, K/64, ...}): a box of two
// 64-column K blocks of box_rows rows is one request (the CTA-pair stages).
// [K][N] weight as a 3-D map (64 columns, k, 64-column block): one box of
// 64 columns x k_rows rows x blocks blocks, 128-byte swizzled rows of k.
static int make_map_mn(CUtensorMap *map, const void *ptr, const cuuint64_t *dims, const cuuint64_t *strides,
                       uint32_t k_rows, uint32_t blocks)
{
    auto fn = encode_fn();
    if (!fn) return set_error(RC_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint32_t box[3] = {64, k_rows, blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3u, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(RC_ERR_INVALID, "tensor map encoding failed (CUresult %d)", (int)r);
    return RC_OK;
}
static int make_map_k2(CUtensorMap *map, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                       uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return set_error(RC_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint32_t box[4] = {64, box_rows, (cuuint32_t)KSUB2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(RC_ERR_INVALID, "tensor map encoding failed (CUresult %d)", (int)r);
    return RC_OK;
}

// Tuning knob, read once from the environment: RC_GEMM_PAIRS=0 keeps the
// one-CTA kernel even where the CTA-pair form applies.
static std::atomic<int> g_skip_row{-1};   // ag_gemm_debug_skip_piece

static bool pair_tiles_enabled()
{
    static const bool v = [] {
        const char *e = getenv("RC_GEMM_PAIRS");
        return !(e && e[0] == '0' && e[1] == 0);
    }();
    return v;
}

static bool overlap(const void *a, size_t an, const void *b, size_t bn)
{
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bn && b0 < a0 + an;
}

} // namespace ag
} // namespace rc

static int ag_gemm_run(const void *a_shards, size_t a_stride, void *a_gathered, const void *B, int b_layout, void *C,
                       int P, int rank, int M_r, int N, int K, void *ws, size_t ws_bytes, void *stream)
{
    using namespace rc;
    using namespace rc::ag;
    if (P < 1 || P > RC_MAX_P) return set_error(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (rank < 0 || rank >= P) return set_error(RC_ERR_INVALID, "rank %d outside 0..P-1", rank);
    if (M_r <= 0 || N <= 0 || K <= 0 || M_r % BM || N % BN || K % BK)
        return set_error(RC_ERR_INVALID, "need M_r %% %d == 0, N %% %d == 0, K %% %d == 0 (got %d, %d, %d)", BM, BN, BK,
                         M_r, N, K);
    if (!a_shards || !a_gathered || !B || !C) return set_error(RC_ERR_INVALID, "null pointer");
    if (b_layout != RC_B_NK && b_layout != RC_B_KN) return set_error(RC_ERR_INVALID, "unknown B layout %d", b_layout);
    if (((uintptr_t)a_shards | (uintptr_t)a_gathered | (uintptr_t)B | (uintptr_t)C | a_stride) & 15u)
        return set_error(RC_ERR_INVALID, "pointers and a_stride must be 16-byte aligned");
    const size_t shard_bytes = (size_t)M_r * K * 2;
    if (P > 1 && a_stride < shard_bytes) return set_error(RC_ERR_INVALID, "a_stride below a shard's bytes");
    const size_t M = (size_t)P * M_r;
    const size_t ag_bytes = M * K * 2, b_bytes = (size_t)N * K * 2, c_bytes = M * N * 2;
    const size_t sh_span = (size_t)(P - 1) * a_stride + shard_bytes;
    if (overlap(a_gathered, ag_bytes, C, c_bytes) || overlap(a_gathered, ag_bytes, a_shards, sh_span) ||
        overlap(a_gathered, ag_bytes, B, b_bytes) || overlap(C, c_bytes, a_shards, sh_span) ||
        overlap(C, c_bytes, B, b_bytes))
        return set_error(RC_ERR_INVALID, "outputs overlap each other or an input");
    if (M > (1u << 31) || (size_t)N > (1u << 31)) return set_error(RC_ERR_INVALID, "dimensions too large");

    Params p{};
    p.a_shards = (const char *)a_shards;
    p.a_stride = a_stride;
    p.a_gathered = (char *)a_gathered;
    p.C = (char *)C;
    p.P = P;
    p.rank = rank;
    p.M_r = M_r;
    p.N = N;
    p.K = K;
    p.g_total_m = (int)(M / BM);
    p.g_per_pe = M_r / BM;
    p.units = p.g_total_m * (BM / PIECE_ROWS);
    p.st32 = (((uintptr_t)C | (size_t)N * 2) & 31u) == 0;
    p.b_kn = b_layout == RC_B_KN;
    int sm_count = 0;
    int rc_ = prepare_workspace_ext(ws, ws_bytes, (size_t)p.units, &p.hdr, &p.flags, &sm_count, &p.timeout_ns);
    if (rc_) return rc_;
    const bool pairs = M_r % PM == 0 && K % BK2 == 0 && sm_count >= 2 && pair_tiles_enabled();
    const size_t sh_stride = P > 1 ? a_stride : shard_bytes;

    CUtensorMap map_ag, map_sh, map_b;
    if (pairs) {
        const cuuint64_t dag[3] = {64, (cuuint64_t)M, (cuuint64_t)K / 64};
        const cuuint64_t sag[2] = {(cuuint64_t)K * 2, 128};
        if ((rc_ = make_map_k2(&map_ag, a_gathered, 3, dag, sag, HM))) return rc_;
        const cuuint64_t dsh[4] = {64, (cuuint64_t)M_r, (cuuint64_t)K / 64, (cuuint64_t)P};
        const cuuint64_t ssh[3] = {(cuuint64_t)K * 2, 128, (cuuint64_t)sh_stride};
        if ((rc_ = make_map_k2(&map_sh, a_shards, 4, dsh, ssh, HM))) return rc_;
        if (p.b_kn) {   // [K][N]: (64 columns, k, 64-column block), box 64 x BK2 x 2
            const cuuint64_t db[3] = {64, (cuuint64_t)K, (cuuint64_t)N / 64};
            const cuuint64_t sb[2] = {(cuuint64_t)N * 2, 128};
            if ((rc_ = make_map_mn(&map_b, B, db, sb, BK2, HN / 64))) return rc_;
        } else {
            const cuuint64_t db[3] = {64, (cuuint64_t)N, (cuuint64_t)K / 64};
            const cuuint64_t sb[2] = {(cuuint64_t)K * 2, 128};
            if ((rc_ = make_map_k2(&map_b, B, 3, db, sb, HN))) return rc_;
        }
    } else {
        {
            cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
            cuuint64_t strides[1] = {(cuuint64_t)K * 2};
            if ((rc_ = make_map(&map_ag, a_gathered, 2, dims, strides, BM))) return rc_;
        }
        {
            cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)M_r, (cuuint64_t)P};
            cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)sh_stride};
            if ((rc_ = make_map(&map_sh, a_shards, 3, dims, strides, BM))) return rc_;
        }
        if (p.b_kn) {   // [K][N]: (64 columns, k, 64-column block), box 64 x BK x 4
            const cuuint64_t db[3] = {64, (cuuint64_t)K, (cuuint64_t)N / 64};
            const cuuint64_t sb[2] = {(cuuint64_t)N * 2, 128};
            if ((rc_ = make_map_mn(&map_b, B, db, sb, BK, BN / 64))) return rc_;
        } else {
            cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
            cuuint64_t strides[1] = {(cuuint64_t)K * 2};
            if ((rc_ = make_map(&map_b, B, 2, dims, strides, BN))) return rc_;
        }
    }

    p.skip_row = g_skip_row.exchange(-1);
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(k_ag_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(k_ag_gemm2, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM2_BYTES);
    });
    if (attr_err != cudaSuccess)
        return set_error(RC_ERR_CUDA, "shared-memory attribute: %s", cudaGetErrorString(attr_err));
    cudaError_t e;
    if (pairs) {
        p.total_m = (int)(M / PM);
        p.tiles_per_pe = M_r / PM;
        p.n_tiles = N / PN;
        p.total_tiles = p.total_m * p.n_tiles;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = SMEM2_BYTES;
        cfg.stream = (cudaStream_t)stream;
        cfg.gridDim = dim3(2);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, (const void *)k_ag_gemm2, &cfg);
        if (e != cudaSuccess) return set_error(RC_ERR_CUDA, "cluster occupancy query: %s", cudaGetErrorString(e));
        if (clusters < 1) return set_error(RC_ERR_UNSUPPORTED, "no CTA pair of the GEMM fits on the GPU");
        if (clusters > p.total_tiles) clusters = p.total_tiles;
        cfg.gridDim = dim3(2 * (unsigned)clusters);
        // Every consumer may wait on ready flags that another CTA's gather
        // producer sets: ask for co-residency (cooperative launch); the grid is
        // sized to the clusters that fit at once, so a runtime that refuses the
        // attribute for clusters still gets every CTA resident.
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, k_ag_gemm2, map_ag, map_sh, map_b, p);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            cfg.numAttrs = 0;
            e = cudaLaunchKernelEx(&cfg, k_ag_gemm2, map_ag, map_sh, map_b, p);
        }
    } else {
        p.total_m = (int)(M / BM);
        p.tiles_per_pe = M_r / BM;
        p.n_tiles = N / BN;
        p.total_tiles = p.total_m * p.n_tiles;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ag_gemm, THREADS, SMEM_BYTES);
        if (e != cudaSuccess) return set_error(RC_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
        if (per_sm < 1) return set_error(RC_ERR_UNSUPPORTED, "the GEMM block does not fit on an SM");
        int grid = sm_count * per_sm;
        if (grid > p.total_tiles) grid = p.total_tiles;
        void *args[] = {(void *)&map_ag, (void *)&map_sh, (void *)&map_b, (void *)&p};
        e = cudaLaunchCooperativeKernel((const void *)k_ag_gemm, dim3((unsigned)grid), dim3(THREADS), args,
                                        (size_t)SMEM_BYTES, (cudaStream_t)stream);
    }
    if (e != cudaSuccess) return set_error(RC_ERR_CUDA, "ag_gemm launch: %s", cudaGetErrorString(e));
    return RC_OK;
}

extern "C" int ag_gemm(const void *a_shards, size_t a_stride, void *a_gathered, const void *B, void *C, int P,
                       int rank, int M_r, int N, int K, void *stream)
{
    return ag_gemm_run(a_shards, a_stride, a_gathered, B, RC_B_NK, C, P, rank, M_r, N, K, nullptr, 0, stream);
}

extern "C" int ag_gemm_kn(const void *a_shards, size_t a_stride, void *a_gathered, const void *B, void *C, int P,
                          int rank, int M_r, int N, int K, void *stream)
{
    return ag_gemm_run(a_shards, a_stride, a_gathered, B, RC_B_KN, C, P, rank, M_r, N, K, nullptr, 0, stream);
}

extern "C" int ag_gemm_ex(const void *a_shards, size_t a_stride, void *a_gathered, const void *B, int b_layout,
                          void *C, int P, int rank, int M_r, int N, int K, void *workspace, size_t ws_bytes,
                          void *stream)
{
    if (!workspace) return rc::set_error(RC_ERR_INVALID, "null workspace");
    return ag_gemm_run(a_shards, a_stride, a_gathered, B, b_layout, C, P, rank, M_r, N, K, workspace, ws_bytes,
                       stream);
}

extern "C" int ag_gemm_debug_skip_piece(int row)
{
    if (row < -1) return rc::set_error(RC_ERR_INVALID, "row %d below -1", row);
    rc::ag::g_skip_row.store(row);
    return RC_OK;
}

// Header + one ready flag per gather unit (PIECE_ROWS rows of A_g).
extern "C" size_t ag_gemm_workspace_bytes(int P, int M_r)
{
    using namespace rc::ag;
    if (P < 1 || P > RC_MAX_P || M_r <= 0 || M_r % BM) return 0;
    const size_t units = (size_t)P * (size_t)(M_r / BM) * (BM / PIECE_ROWS);
    return sizeof(rc::WsHeader) + units * 4;
}
