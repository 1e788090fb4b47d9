// ring_kernels.cu -- the ring step engine (all-reduce, reduce-scatter,
// all-gather) and the right-shift copy kernel.
//
// One persistent launch runs a whole collective.  Thread block (r, j) plays
// logical rank r for slice j of every chunk: slice j of the chunks forms an
// independent ring of P blocks with its own signal rows, so S slices give
// P*S blocks that all stream at once.  The launch is cooperative, so every
// block is resident and a block spinning on its left neighbour cannot starve
// it.
//
// Ring schedule ("全归约 3：Ring——每步大小恒定", section "走读"): global
// step g waits on signal row g written by the left neighbour (row 0 of the
// all-reduce and reduce-scatter is satisfied at launch: the inputs are already
// in place), moves one slice of one chunk, then notifies row g+1 of the right
// neighbour.  Reduce-scatter round s adds the left neighbour's chunk
// (r-s-2+P)%P into the local chunk of that index; all-gather round t copies
// the left neighbour's chunk (r-1-t+P)%P.  Signal rows are monotonic: a
// notify stores the launch's epoch (one more than the launches completed on
// the workspace) and a wait tests "reached the epoch", so rows never need
// resetting between calls.
//
// Data movement: reduce-scatter steps stream 32-byte vectors through
// registers (two loads, one hop add, one store per vector); all-gather steps
// move their slice with 32-byte vector copies (all-reduce) or with bulk (TMA)
// copies staged in shared memory (standalone all-gather), as RingParams::ag_bulk
// says.
//
// Why no extra guard against overwriting data a neighbour still reads: rank
// r reads its left neighbour's chunk (r-s-2) in round s; the left neighbour
// rewrites that chunk only in all-gather round s (global step P-1+s), and
// reaching that step needs a chain of P-1 notifies around the ring that ends
// with rank r's notify of step s, issued after rank r's loads of step s.
#include "internal.h"
#include "dev.cuh"
#include "ring_common.cuh"
#include "ringcoll.h"
#include "tc.cuh"

namespace rc {

// ------------------------------------------------------------ bulk all-gather copies
// An all-gather step copies one slice of a chunk from the left neighbour's
// slot into the own slot.  With p.ag_bulk, thread 0 moves the 16-byte
// aligned body of that range with bulk (TMA) copies through kAgStages
// shared-memory buffers: loads (global -> shared, completing on one mbarrier
// per stage) run up to kAgStages-1 pieces ahead of the stores (shared ->
// global, bulk groups), while warp 1 copies the unaligned head and tail
// element-wise.
struct BulkCtx {
    uint32_t buf;    // shared address of stage 0
    uint32_t bar;    // shared address of the mbarrier of stage 0 (8 bytes per stage)
    uint32_t phase;  // parity bit per stage (thread 0)
};

// Waits for a stage's load.  A load that has not landed after timeout_ns
// records RC_ERR_TIMEOUT (the launch then stops at its next step) and is
// waited for once more, so no copy still targets shared memory when the
// block exits; false if it failed.
__device__ bool bulk_bar_wait(uint32_t bar, uint32_t parity, const RingParams &p, int r, int g, int j)
{
    uint64_t t0 = 0;
    bool late = false;
    for (uint32_t it = 0;; ++it) {
        if (tc::mbar_try_wait(bar, parity)) return !late;
        if ((it & 255u) == 255u) {
            const uint64_t now = global_timer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > p.timeout_ns) {
                if (late) return false;
                if (atomicCAS(&p.hdr->status, 0u, (unsigned)RC_ERR_TIMEOUT) == 0u) {
                    p.hdr->err_rank = (uint32_t)r;
                    p.hdr->err_step = (uint32_t)g;
                    p.hdr->err_slice = (uint32_t)j;
                }
                late = true;
                t0 = now;
            }
        }
    }
}

// Thread 0: dst[0, bytes) = src[0, bytes), both 16-byte aligned, bytes a
// multiple of 16.  Runs after this thread's acquire of the step's signal
// row: the proxy fence orders that acquire before the async-proxy loads
// and stores.  On return every store has completed and a second proxy fence
// orders them before the generic-proxy release of the next notify.
__device__ bool bulk_copy_body(char *dst, const char *src, size_t bytes, BulkCtx &bc, uint64_t pol_src,
                               uint64_t pol_dst, const RingParams &p, int r, int g, int j)
{
    constexpr size_t SB = kAgStageBytes;
    const size_t np = (bytes + SB - 1) / SB;
    tc::fence_proxy_async_global();
    const size_t pre = np < (size_t)kAgStages ? np : (size_t)kAgStages;
    for (size_t i = 0; i < pre; ++i) {
        const uint32_t len = (uint32_t)(bytes - i * SB < SB ? bytes - i * SB : SB);
        tc::mbar_expect_tx(bc.bar + 8u * (uint32_t)i, len);
        tc::bulk_g2s_hint(bc.buf + (uint32_t)(i * SB), src + i * SB, len, bc.bar + 8u * (uint32_t)i, pol_src);
    }
    bool ok = true;
    for (size_t i = 0; i < np; ++i) {
        const uint32_t s = (uint32_t)(i % kAgStages);
        const bool landed = bulk_bar_wait(bc.bar + 8u * s, (bc.phase >> s) & 1u, p, r, g, j);
        bc.phase ^= 1u << s;
        if (!landed) ok = false;
        if (!ok) continue;   // drain the loads already issued; issue nothing more
        const size_t off = i * SB;
        const uint32_t len = (uint32_t)(bytes - off < SB ? bytes - off : SB);
        tc::bulk_s2g_hint(dst + off, bc.buf + s * (uint32_t)SB, len, pol_dst);
        tc::bulk_commit();
        const size_t nx = i - 1 + kAgStages;   // next piece for the stage of piece i-1
        if (i >= 1 && nx < np) {
            tc::bulk_wait_read1();              // the store of piece i-1 has read its stage
            const uint32_t t = (uint32_t)(nx % kAgStages);
            const uint32_t nlen = (uint32_t)(bytes - nx * SB < SB ? bytes - nx * SB : SB);
            tc::mbar_expect_tx(bc.bar + 8u * t, nlen);
            tc::bulk_g2s_hint(bc.buf + t * (uint32_t)SB, src + nx * SB, nlen, bc.bar + 8u * t, pol_src);
        }
    }
    tc::bulk_wait_all();
    tc::fence_proxy_async_global();
    return ok;
}

// All threads: dst[0, n) = src[0, n) for an all-gather step.  Without bulk
// copies (or when dst and src differ in their offset modulo 16) the block
// streams it with 32-byte vectors; LAST marks the launch's final write of
// the range (evict-first).
template <int ES, bool LAST>
__device__ __forceinline__ void ag_copy(char *dst, const char *src, size_t n, BulkCtx &bc, const RingParams &p,
                                        int r, int g, int j, int *abort_flag)
{
    if (!p.ag_bulk || (((uintptr_t)dst ^ (uintptr_t)src) & 15u) != 0) {
        copy_range<ES, kRingThreads, LAST ? kStEvictFirst : kStNormal>(dst, src, n);
        return;
    }
    const size_t mis = (uintptr_t)dst & 15u;   // a multiple of ES (slots are element-aligned)
    size_t head = mis ? (16 - mis) / ES : 0;
    if (head > n) head = n;
    const size_t body = ((n - head) * ES) & ~(size_t)15;
    const size_t done = head + body / ES;
    if (threadIdx.x == 0) {
        if (body && !bulk_copy_body(dst + head * ES, src + head * ES, body, bc, tc::policy_evict_first(),
                                    LAST ? tc::policy_evict_first() : tc::policy_evict_normal(), p, r, g, j))
            *abort_flag = 1;
    } else if (threadIdx.x >= 32 && threadIdx.x < 64) {
        const size_t lane = threadIdx.x - 32;
        for (size_t i = lane; i < head; i += 32) {
            if (ES == 2) st_u16(dst + 2 * i, ld_cg_u16(src + 2 * i));
            else st_u32(dst + 4 * i, ld_cg_u32(src + 4 * i));
        }
        for (size_t i = done + lane; i < n; i += 32) {
            if (ES == 2) st_u16(dst + 2 * i, ld_cg_u16(src + 2 * i));
            else st_u32(dst + 4 * i, ld_cg_u32(src + 4 * i));
        }
    }
}

// ------------------------------------------------------------ the step engine
// Segments: when one step's live data (P chunks) would not fit in L2, each
// slice ring runs all its steps on segment 0 of the chunks, then segment 1,
// and so on (segment q of chunk k is the same element range in every chunk,
// so every element keeps its ring order).  Segment q signals with the value
// E0 + q + 1 on the same rows (E0: the epoch before the launch), so values
// stay monotonic across segments and launches; the launch advances the epoch
// by the number of segments.
//
// MODE_RS_BIDIR (the bidirectional reduce-scatter of "Pallas TPU Distributed
// Collectives 复习文档", section 4): block (h, r, j) runs half h of every
// chunk (h = 0: the top half [0, c/2), which travels left; h = 1: the bottom
// half [c/2, c), which travels right) as its own ring.  In step s = 0..P-2
// rank r adds the partial its upstream neighbour (right for the top, left for
// the bottom) holds for chunk (r+1+s) resp. (r-1-s) to its own contribution.
// Step P-2 completes chunk (r-1) resp. (r+1) -- the chunk of the very
// neighbour this block notifies -- and stores it straight into that rank's
// out slot: the page's last hop only moves the finished sum to its owner, so
// folding it into the store saves a read and a write of every half and one
// signalled step.  Each chunk half is written once, so no buffer is ever
// overwritten while read.
// SERIAL: the barrier-injection debug variant (RingParams::debug_serial); a
// separate instantiation, so the normal kernels carry none of its state.
template <int DT, int MODE, bool SERIAL>
__global__ void __launch_bounds__(kRingThreads, RC_RING_MIN_BLOCKS) k_ring(const RingParams p)
{
    constexpr size_t ES = DT == 1 ? 2 : 4;
    constexpr bool BIDIR = MODE == MODE_RS_BIDIR;
    const int P = p.P, S = p.S;
    const int rs = (int)(blockIdx.x / (unsigned)S), j = (int)(blockIdx.x % (unsigned)S);
    const int h = BIDIR ? rs / P : 0;              // half (bidirectional mode only)
    const int r = BIDIR ? rs % P : rs;
    const int left = (r - 1 + P) % P, right = (r + 1) % P;
    const int from = (BIDIR && h == 0) ? right : left; // whose data this block pulls
    const int to = (BIDIR && h == 0) ? left : right;   // whom this block notifies
    // The abort word is the header's pad[0]: a launch that gives up stores its epoch there.
    uint32_t *abort_word = &p.hdr->pad[0];
    const int nsteps = MODE == MODE_ALLREDUCE ? 2 * (P - 1) : P - 1;

    // State only thread 0 uses (signal rows, step stamps) lives in shared
    // memory so it does not hold registers through the streaming loops.
    __shared__ uint32_t s_epoch0;
    __shared__ int s_abort;
    __shared__ const uint32_t *s_my_rows;   // [steps][P] signal words of (rank r, slice j, half h)
    __shared__ uint32_t *s_to_rows;         // the same for the block this one notifies
    __shared__ unsigned long long *s_stamp; // step stamps of this block, or null
    // Bulk-copy staging is dynamic shared memory, present only in launches that
    // run all-gather steps with bulk copies (ring_dyn_smem): the other modes
    // leave that space to L1.
    extern __shared__ __align__(128) unsigned char s_bulk[];
    __shared__ __align__(8) uint64_t s_bulk_bar[kAgStages];
    BulkCtx bc{tc::smem_u32(s_bulk), tc::smem_u32(s_bulk_bar), 0u};
    if (threadIdx.x == 0) {
        if (p.ag_bulk) {
            for (int s = 0; s < kAgStages; ++s) tc::mbar_init(bc.bar + 8u * (uint32_t)s, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        s_epoch0 = ld_relaxed_gpu(&p.hdr->epoch);
        s_abort = 0;
        s_my_rows = p.sig + (((size_t)j * P + r) * (size_t)p.rows + (size_t)h * nsteps) * P;
        s_to_rows = p.sig + (((size_t)j * P + to) * (size_t)p.rows + (size_t)h * nsteps) * P;
        s_stamp = (p.trace && (size_t)(blockIdx.x + 1) * nsteps * 3 <= p.trace_words)
                      ? p.trace + (size_t)blockIdx.x * nsteps * 3
                      : nullptr;
    }
    __syncthreads();
    if (p.stagger_groups > 1) {
        // Phase-shifted slice rings (RingParams::stagger_*): every block of
        // slice j, i.e. the whole ring, starts (j % groups) * stagger_ns later.
        const unsigned g = (unsigned)j % (unsigned)p.stagger_groups;
        if (g && threadIdx.x == 0) {
            const uint64_t t0 = global_timer_ns(), d = (uint64_t)g * p.stagger_ns;
            while (global_timer_ns() - t0 < d) __nanosleep(128);
        }
        __syncthreads();
    }
    const uint32_t E0 = s_epoch0;
    const uint32_t E = E0 + 1u;   // identifies this launch (abort word)
    const size_t c = p.chunk;
    const size_t cs = p.chunk_stride;   // elements from one chunk's start to the next (>= c)
    const size_t half = c / 2;
    const size_t range_lo = BIDIR ? (h == 0 ? 0 : half) : 0;     // element range of this block's ring
    const size_t range_n = BIDIR ? (h == 0 ? half : c - half) : c;
    char *my_slot = p.data + (size_t)r * p.data_stride;
    const char *from_slot = p.data + (size_t)from * p.data_stride;
    constexpr int T = kRingThreads;
    uint32_t meet_round = 0;   // debug grid barriers passed (RC_DEBUG_SERIAL)

    for (int q = 0; q < p.segments; ++q) {
        const size_t seg_lo = range_lo + slice_begin(range_n, q, p.segments);
        const size_t seg_n = range_lo + slice_begin(range_n, q + 1, p.segments) - seg_lo;
        const size_t lo = seg_lo + slice_begin(seg_n, j, S);
        const size_t n = seg_lo + slice_begin(seg_n, j + 1, S) - lo;
        const uint32_t V = E0 + 1u + (uint32_t)q; // signal value of this segment

        if (MODE == MODE_ALL_GATHER) {
            // Prologue: the own shard goes to chunk r of the own output slot,
            // then the right neighbour's first row says it may be read.
            copy_range<ES, T, kStNormal>(my_slot + ((size_t)r * cs + lo) * ES, p.in + (size_t)r * p.in_stride + lo * ES,
                                         n);
            __syncthreads();
            if (threadIdx.x == 0) st_release_gpu(&s_to_rows[r], V);
        }

        // Step stamps (%globaltimer, thread 0, first segment): per block and
        // step, the start of the wait, its end, and the end of the step.
        for (int g = 0; g < nsteps; ++g) {
            if (threadIdx.x == 0 && s_stamp && q == 0) s_stamp[3 * g] = global_timer_ns();
            if (g > 0 || MODE == MODE_ALL_GATHER) {
#if RC_RING_PREFETCH
                // Standalone reduce-scatter rounds: the own chunk's input does not
                // depend on the left neighbour, so while thread 0 waits for its
                // signal the other threads pull the first lines of this block's
                // slice of it into L2.  (Measured on GB300 at P=8 x 64 MiB bf16:
                // 0.1379 -> 0.1355 ms; in the all-reduce, whose all-gather data
                // also competes for L2, it costs 0.5-2 %, so it is off there.)
                if (MODE == MODE_REDUCE_SCATTER && g < P - 1 && threadIdx.x > 0 && threadIdx.x <= RC_RING_PREFETCH) {
                    const int k = (r - g - 2 + P) % P;
                    const size_t line = (size_t)(threadIdx.x - 1) * 128;
                    if (line < n * ES) prefetch_l2_line(my_slot + ((size_t)k * cs + lo) * ES + line);
                }
#endif
                if (threadIdx.x == 0 &&
                    !wait_row(&s_my_rows[(size_t)g * P + from], V, E, p, r, g, j, abort_word))
                    s_abort = 1;
                __syncthreads();
                if (s_abort) break;
            }
            if (threadIdx.x == 0 && s_stamp && q == 0) s_stamp[3 * g + 1] = global_timer_ns();
            const bool last = g == nsteps - 1; // nothing reads this step's output again in this launch
            if (MODE == MODE_ALL_GATHER) {
                const int k = (r - 1 - g + P) % P;
                const size_t off = ((size_t)k * cs + lo) * ES;
                if (last)
                    ag_copy<ES, true>(my_slot + off, from_slot + off, n, bc, p, r, g, j, &s_abort);
                else
                    ag_copy<ES, false>(my_slot + off, from_slot + off, n, bc, p, r, g, j, &s_abort);
            } else if (BIDIR) {
                // partial for chunk k: the upstream neighbour's partial (+) own contribution
                const int k = h == 0 ? (r + 1 + g) % P : (r - 1 - g + 2 * P) % P;
                const size_t off = ((size_t)k * cs + lo) * ES;
                // The partial read here is dead afterwards (no one reads or
                // rewrites it again): its lines are dropped from step s = 1 on.
                if (last) // k == to: the finished sum goes to its owner's out slot
                    add_range<DT, T, kStNormal, false>(p.out + (size_t)k * p.out_stride + lo * ES, from_slot + off,
                                                my_slot + off, n, p.discard && g >= 1);
                else
                    add_range<DT, T, kStEvictLast, false>(my_slot + off, from_slot + off, my_slot + off, n,
                                                   p.discard && g >= 1);
            } else if (g < P - 1) {
                const int s = g;
                const int k = (r - s - 2 + P) % P; // recv_add_idx == left_send_idx
                const size_t off = ((size_t)k * cs + lo) * ES;
                char *own = my_slot + off;
                char *dst = (MODE == MODE_REDUCE_SCATTER && s == P - 2)
                                ? p.out + (size_t)r * p.out_stride + lo * ES
                                : own;
                // From reduce-scatter step s = 1 on, the left chunk read here is the partial sum the
                // left neighbour wrote in round s-1; no one reads it again before
                // the left neighbour overwrites it (all-gather round s), so its
                // dirty L2 lines are dropped instead of being written back.  The
                // drops precede this step's notify, which orders them before that
                // overwrite (it needs P-1 notifies round the ring, this one last).
                // Rounds 0..P-3 write partial sums that the right neighbour reads
                // next round and then drops: keep them in L2 (evict_last).  The last
                // round writes the reduced chunk (read by the all-gather, or the output).
                const bool drop = p.discard && s >= 1;
                if (p.discard && s < P - 2)
                    add_range<DT, T, kStEvictLast, MODE == MODE_ALLREDUCE>(dst, from_slot + off, own, n, drop);
                else
                    add_range<DT, T, kStNormal, MODE == MODE_ALLREDUCE>(dst, from_slot + off, own, n, drop);
            } else {
                const int t = g - (P - 1);
                const int k = (r - 1 - t + P) % P;
                const size_t off = ((size_t)k * cs + lo) * ES;
                if (last)
                    ag_copy<ES, true>(my_slot + off, from_slot + off, n, bc, p, r, g, j, &s_abort);
                else
                    ag_copy<ES, false>(my_slot + off, from_slot + off, n, bc, p, r, g, j, &s_abort);
            }
            if (g + 1 < nsteps) {
                __syncthreads(); // every thread's loads, stores and drops of this step precede the release
                if (s_abort) break;
                if (threadIdx.x == 0 && !(r == p.skip_rank && g == p.skip_step))
                    st_release_gpu(&s_to_rows[(size_t)(g + 1) * P + r], V);
            }
            if (threadIdx.x == 0 && s_stamp && q == 0) s_stamp[3 * g + 2] = global_timer_ns();
            if constexpr (SERIAL) {
                grid_meet(p, ++meet_round, E, abort_word, r, g, j, &s_abort);
                if (s_abort) break;
            }
        }
        if (s_abort) break;
    }

    // Epilogue: the last block to finish publishes the new epoch.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&p.hdr->done, 1u);
        if (prev == gridDim.x - 1) {
            p.hdr->done = 0;
            p.hdr->pad[1] = 0;   // debug grid-barrier counter
            st_relaxed_gpu(&p.hdr->epoch, E0 + (uint32_t)p.segments);
        }
    }
}

// ------------------------------------------------------------ right shift
// dst_r = src_{(r-1+P)%P}: blockIdx.y is the destination rank, blocks along x
// split the slot into contiguous pieces.
template <int ES>
__global__ void __launch_bounds__(256) k_ppermute(const char *src, size_t ss, char *dst, size_t ds, int P, size_t n)
{
    const int r = blockIdx.y;
    const int left = (r - 1 + P) % P;
    const char *s = src + (size_t)left * ss;
    char *d = dst + (size_t)r * ds;
    // contiguous pieces of whole 256-byte runs (64 or 128 elements)
    constexpr size_t G = 256 / ES;
    const size_t runs = (n + G - 1) / G;
    const size_t per = (runs + gridDim.x - 1) / gridDim.x;
    const size_t b0 = min(n, per * blockIdx.x * G), b1 = min(n, per * (blockIdx.x + 1) * G);
    if (b0 < b1) copy_range<ES, 256, kStEvictFirst>(d + b0 * ES, s + b0 * ES, b1 - b0);
}

// ------------------------------------------------------------ L2 step-rate probe
// The ring's own streaming loops, run `reps` times over one range: with the
// range's buffers resident in L2 this measures how fast an all-gather step
// (copy: 1 read + 1 write) or a reduce-scatter step (add: 2 reads + 1 write)
// can move data through L2, the ceiling of every ring step after the first.
// Block i of the grid takes bytes [i*per, (i+1)*per) of the range.
template <bool ADD>
__global__ void __launch_bounds__(kRingThreads, RC_RING_MIN_BLOCKS)
    k_l2_rate(char *dst, const char *a, const char *b, size_t bytes, size_t per, int reps)
{
    const size_t lo = (size_t)blockIdx.x * per;
    if (lo >= bytes) return;
    const size_t n = (bytes - lo < per ? bytes - lo : per) / 4;
    for (int i = 0; i < reps; ++i) {
        if (ADD)
            add_range<0, kRingThreads, kStNormal>(dst + lo, a + lo, b + lo, n, false);
        else
            copy_range<4, kRingThreads, kStNormal>(dst + lo, a + lo, n);
        __syncthreads();
    }
}

// ------------------------------------------------------------ host launchers
template <int DT, bool SERIAL>
static const void *ring_fn_mode(int mode)
{
    switch (mode) {
    case MODE_ALLREDUCE: return (const void *)k_ring<DT, MODE_ALLREDUCE, SERIAL>;
    case MODE_REDUCE_SCATTER: return (const void *)k_ring<DT, MODE_REDUCE_SCATTER, SERIAL>;
    case MODE_ALL_GATHER: return (const void *)k_ring<DT, MODE_ALL_GATHER, SERIAL>;
    default: return (const void *)k_ring<DT, MODE_RS_BIDIR, SERIAL>;
    }
}

static const void *ring_fn(int dtype, int mode, bool serial = false)
{
    if (serial) {
        switch (dtype) {
        case 0: return ring_fn_mode<0, true>(mode);
        case 1: return ring_fn_mode<1, true>(mode);
        default: return ring_fn_mode<2, true>(mode);
        }
    }
    switch (dtype) {
    case 0: return ring_fn_mode<0, false>(mode);
    case 1: return ring_fn_mode<1, false>(mode);
    default: return ring_fn_mode<2, false>(mode);
    }
}

// Dynamic shared memory of a ring launch: the bulk-copy staging, for modes
// with all-gather steps when bulk copies are on.
static size_t ring_dyn_smem(int mode, int ag_bulk)
{
    return ag_bulk && (mode == MODE_ALLREDUCE || mode == MODE_ALL_GATHER) ? (size_t)kAgStages * kAgStageBytes : 0;
}

cudaError_t ring_max_coresident(int dtype, int threads, int device, int *blocks)
{
    // every mode instantiation has the same register budget (launch bounds); take the minimum
    int sms = 0, best = 1 << 30;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    for (int mode = 0; mode < 8; ++mode) {   // four modes, normal and serial-debug variants
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ring_fn(dtype, mode & 3, mode >= 4), threads,
                                                          ring_dyn_smem(mode & 3, 1));
        if (e != cudaSuccess) return e;
        if (per_sm < best) best = per_sm;
    }
    *blocks = best * sms;
    return cudaSuccess;
}

cudaError_t launch_ring(const RingParams &p, int dtype, int threads, cudaStream_t st)
{
    RingParams copy = p;
    if (copy.chunk_stride == 0) copy.chunk_stride = copy.chunk;   // chunks back to back
    void *args[] = {(void *)&copy};
    const unsigned blocks = (unsigned)(p.P * p.S) * (p.mode == MODE_RS_BIDIR ? 2u : 1u);
    return cudaLaunchCooperativeKernel(ring_fn(dtype, copy.mode, copy.debug_serial != 0), dim3(blocks),
                                       dim3((unsigned)threads), args, ring_dyn_smem(copy.mode, copy.ag_bulk), st);
}

cudaError_t launch_l2_rate(char *dst, const char *a, const char *b, size_t bytes, int reps, int add, int sm_count,
                           cudaStream_t st)
{
    // the ring's launch shape: RC_RING_MIN_BLOCKS blocks of kRingThreads per SM
    const unsigned blocks = (unsigned)(sm_count * RC_RING_MIN_BLOCKS);
    size_t per = (bytes + blocks - 1) / blocks;
    per = (per + 255) & ~(size_t)255;   // whole 256-byte runs per block
    if (add)
        k_l2_rate<true><<<blocks, kRingThreads, 0, st>>>(dst, a, b, bytes, per, reps);
    else
        k_l2_rate<false><<<blocks, kRingThreads, 0, st>>>(dst, a, b, bytes, per, reps);
    return cudaGetLastError();
}

cudaError_t launch_ppermute(const char *src, size_t src_stride, char *dst, size_t dst_stride, int P, size_t n,
                            int esize, int sm_count, cudaStream_t st)
{
    // About RC_PPERMUTE_BLOCKS_PER_SM blocks per SM in total, at least one per rank.
    const size_t bytes = n * (size_t)esize;
    unsigned bx = (unsigned)(((size_t)RC_PPERMUTE_BLOCKS_PER_SM * (size_t)sm_count + P - 1) / P);
    const size_t max_bx = (bytes + 16383) / 16384; // no block below ~16 KiB
    if (bx > max_bx) bx = (unsigned)max_bx;
    if (bx < 1) bx = 1;
    dim3 grid(bx, (unsigned)P);
    if (esize == 2)
        k_ppermute<2><<<grid, 256, 0, st>>>(src, src_stride, dst, dst_stride, P, n);
    else
        k_ppermute<4><<<grid, 256, 0, st>>>(src, src_stride, dst, dst_stride, P, n);
    return cudaGetLastError();
}

} // namespace rc
