// ring_pair.cu -- the ring step engine with two logical ranks per thread block.
//
// The schedule is the one of k_ring ("全归约 3：Ring——每步大小恒定", section
// "走读"): every rank runs the same 2(P-1) global steps (P-1 for the
// reduce-scatter), reduce-scatter round s adding its left neighbour's chunk
// (r-s-2+P)%P into its own chunk of that index, all-gather round t copying
// the left neighbour's chunk (r-1-t+P)%P.  What changes is where the ranks
// run: thread block (m, j) plays ranks r0 = 2m and r1 = 2m+1 for slice j, so
// the P/2 blocks of a slice form the ring and every other hop stays inside
// one block.
//
// Why.  A ring step's data is already on chip except for the first step, so
// the all-reduce is bound by the rate at which L2 serves reads and writes: a
// reduce-scatter hop writes a partial sum to L2 that the right neighbour reads
// back one step later.  For the hop r0 -> r1 the block keeps the head of
// that partial (p.hand_bytes per block) in shared memory instead, so the
// write, the read and the L2 line drop of that part disappear; the rest of
// the slice, and every hop between blocks, goes through the slots as in
// k_ring.  All-gather hops r0 -> r1 read their source from the same shared
// copy.  The slots still receive every final value.
//
// Order inside a block, per global step g:
//   1. rank r1 does step g.  It needs rank r0's step g-1 output only (shared
//      memory head + slot rest, produced by this block), so it runs before
//      the wait on the previous block.
//   2. __syncthreads, then notify the next block (whose r0 is r1's right
//      neighbour) on signal row g+1.
//   3. wait for the previous block's notify on row g (its r1 is r0's left
//      neighbour); row 0 is satisfied at launch.
//   4. rank r0 does step g, leaving its output head in shared memory for
//      step 1 of the next iteration; __syncthreads.
// Write-after-read safety is the argument of k_ring: rank r0 reads its left
// neighbour's chunk (r0-s-2) in round s, and the left neighbour rewrites it
// in all-gather round s (global step P-1+s); the chain of notifies that
// lets it reach that step starts with this block's notify after step 1 of
// iteration s+1, issued after step 4 of iteration s (program order and a
// __syncthreads).  P = 2 is one block per slice that notifies itself.
#include "internal.h"
#include "dev.cuh"
#include "ring_common.cuh"
#include "ringcoll.h"

namespace rc {

// Shared-memory place of 32-byte vector v of the handed-over head: its two
// 16-byte halves at (v/32)*1024 + (v%32)*16 and 512 bytes later, so the 32
// consecutive vectors of a warp touch 512 contiguous bytes per half.
__device__ __forceinline__ uint32_t hand_off(size_t v) { return (uint32_t)((v >> 5) * 1024 + (v & 31) * 16); }

__device__ __forceinline__ void lds8(uint32_t base, size_t v, uint4 &a, uint4 &b)
{
    const uint32_t o = base + hand_off(v);
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w) : "r"(o)
                 : "memory");
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "r"(o + 512u) : "memory");
}

__device__ __forceinline__ void sts8(uint32_t base, size_t v, const uint4 &a, const uint4 &b)
{
    const uint32_t o = base + hand_off(v);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(o), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w)
                 : "memory");
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(o + 512u), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// Head of a reduce-scatter step, hv 32-byte vectors (a multiple of 32):
// out = a (+) b, with a read from shared memory (A_SM) or global memory,
// b from global memory, and out stored to shared memory (D_SM), to global
// memory (D_GL), or both.  Warp-grouped like add_vec32, including the L2
// drops of a global `a` whose data is dead after this read.
template <int DT, int T, bool A_SM, bool D_SM, bool D_GL, int POL>
__device__ __forceinline__ void head_add(char *dg, uint32_t sm, const char *ag, const char *bg, size_t hv,
                                         bool discard)
{
    constexpr int U = RC_RING_ADD_U;
    const size_t lane = threadIdx.x & 31u;
    size_t vw = threadIdx.x - lane;
    const bool dline = !A_SM && discard && (((uintptr_t)ag & 127u) == 0);
    for (; vw + 31 + (U - 1) * T < hv; vw += U * T) {
        const size_t v = vw + lane;
        uint4 x0[U], x1[U], y0[U], y1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (A_SM)
                lds8(sm, v + u * T, x0[u], x1[u]);
            else
                ld8_ef(ag + (v + u * T) * 32, x0[u], x1[u]);
            ld8_ef(bg + (v + u * T) * 32, y0[u], y1[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint4 z0 = hop_add_v4<DT>(x0[u], y0[u]), z1 = hop_add_v4<DT>(x1[u], y1[u]);
            if (D_SM) sts8(sm, v + u * T, z0, z1);
            if (D_GL) st8<POL>(dg + (v + u * T) * 32, z0, z1);
        }
        if (dline) {
            __syncwarp();
            if (lane < 8 * U) discard_l2_line(ag + (vw + (lane >> 3) * T) * 32 + (lane & 7) * 128);
        }
    }
    if (vw < hv) {   // one partial round (hv is a multiple of 32: whole warps, whole lines)
        const size_t v = vw + lane;
        uint4 x0[U] = {}, x1[U] = {}, y0[U] = {}, y1[U] = {};
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t ok = vw + u * T < hv;   // warp-uniform
            if (A_SM) {
                if (ok) lds8(sm, v + u * T, x0[u], x1[u]);
            } else {
                ld8_ef_if(ag + (v + u * T) * 32, ok, x0[u], x1[u]);
            }
            ld8_ef_if(bg + (v + u * T) * 32, ok, y0[u], y1[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (vw + u * T < hv) {
                const uint4 z0 = hop_add_v4<DT>(x0[u], y0[u]), z1 = hop_add_v4<DT>(x1[u], y1[u]);
                if (D_SM) sts8(sm, v + u * T, z0, z1);
                if (D_GL) st8<POL>(dg + (v + u * T) * 32, z0, z1);
            }
        if (dline) {
            __syncwarp();
            if (lane < 8 * U && vw + (lane >> 3) * T < hv)
                discard_l2_line(ag + (vw + (lane >> 3) * T) * 32 + (lane & 7) * 128);
        }
    }
}

// Head of an all-gather step: out = a over hv vectors, a from shared memory
// (A_SM) or global memory, out to global memory and, with D_SM, also to
// shared memory.
template <int T, bool A_SM, bool D_SM, int POL>
__device__ __forceinline__ void head_copy(char *dg, uint32_t sm, const char *ag, size_t hv)
{
    constexpr int U = 4;
    size_t v = threadIdx.x;
    for (; v + (U - 1) * T < hv; v += U * T) {
        uint4 x0[U], x1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (A_SM)
                lds8(sm, v + u * T, x0[u], x1[u]);
            else
                ld8_ef(ag + (v + u * T) * 32, x0[u], x1[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (D_SM) sts8(sm, v + u * T, x0[u], x1[u]);
            st8<POL>(dg + (v + u * T) * 32, x0[u], x1[u]);
        }
    }
    if (v < hv) {   // one partial round
        uint4 x0[U] = {}, x1[U] = {};
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t ok = v + u * T < hv;
            if (A_SM) {
                if (ok) lds8(sm, v + u * T, x0[u], x1[u]);
            } else {
                ld8_ef_if(ag + (v + u * T) * 32, ok, x0[u], x1[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + u * T < hv) {
                if (D_SM) sts8(sm, v + u * T, x0[u], x1[u]);
                st8<POL>(dg + (v + u * T) * 32, x0[u], x1[u]);
            }
    }
}

// L2 policies of final values: kPolReadNext for data that another rank reads
// from L2 in the next step (kept until that read, which loads it
// evict_first), kPolNoReread for the global copy of a head whose reader takes
// it from shared memory (written back, never read from L2 again).
#ifndef RC_PAIR_POLICIES
#define RC_PAIR_POLICIES 1
#endif
constexpr int kPolReadNext = RC_PAIR_POLICIES ? kStEvictLast : kStNormal;
constexpr int kPolNoReread = RC_PAIR_POLICIES ? kStEvictFirst : kStNormal;

template <int DT, int MODE, bool SERIAL>
__global__ void __launch_bounds__(kPairThreads, RC_PAIR_MIN_BLOCKS) k_ring_pair(const RingParams p)
{
    constexpr size_t ES = DT == 1 ? 2 : 4;
    constexpr int T = kPairThreads;
    constexpr bool BIDIR = MODE == MODE_RS_BIDIR;
    const int P = p.P, S = p.S;
#ifndef RC_PAIR_SPREAD
#define RC_PAIR_SPREAD 1
#endif
    // Block numbering: spread, b = slice * (blocks per slice) + ring block,
    // so consecutive blocks -- which the launch spreads over different SMs --
    // belong to one slice's rings; or b = (ring block) * S + slice, which
    // puts a whole slice ring on one SM when S is the SM count.  Measured on
    // GB300 (P=8 x 64 MiB, 3 x 30 steps): all-reduce 0.1907 -> 0.1903 ms,
    // reduce-scatter unchanged, bidirectional reduce-scatter 0.1210 ->
    // 0.1129 ms with the spread numbering.
    const int per_slice = (BIDIR ? 2 : 1) * (P / 2);
    const int bm = RC_PAIR_SPREAD ? (int)(blockIdx.x % (unsigned)per_slice) : (int)(blockIdx.x / (unsigned)S);
    const int j = RC_PAIR_SPREAD ? (int)(blockIdx.x / (unsigned)per_slice) : (int)(blockIdx.x % (unsigned)S);
    // The bidirectional reduce-scatter runs two rings per slice: half 0 (the
    // top half of every chunk) towards lower ranks, half 1 towards higher
    // ranks; every other mode runs one ring towards higher ranks.
    const int hf = BIDIR ? bm / (P / 2) : 1;
    const int m = BIDIR ? bm % (P / 2) : bm;
    const int r0 = 2 * m, r1 = 2 * m + 1;
    const bool rightward = hf == 1;
    const int rL = rightward ? r1 : r0;                          // fed by its partner in this block
    const int rR = rightward ? r0 : r1;                          // fed by another block
    const int up = rightward ? (r0 - 1 + P) % P : (r1 + 1) % P;  // rR's upstream neighbour (another block)
    const int down = rightward ? (r1 + 1) % P : (r0 - 1 + P) % P; // rL's downstream neighbour (another block)
    uint32_t *abort_word = &p.hdr->pad[0];
    const int nsteps = MODE == MODE_ALLREDUCE ? 2 * (P - 1) : P - 1;
    const size_t row_h = BIDIR ? (size_t)hf * nsteps : 0;       // first signal row of this ring
    // Chunk rank r works on in reduce-scatter step s: (r-s-2) in the
    // one-direction ring; (r-1-s) / (r+1+s) in the bidirectional halves.
    auto chunk_of = [&](int r, int s_) {
        return BIDIR ? (rightward ? (r - 1 - s_ + 2 * P) % P : (r + 1 + s_) % P) : (r - s_ - 2 + 2 * P) % P;
    };

    __shared__ uint32_t s_epoch0;
    __shared__ int s_abort;
    __shared__ const uint32_t *s_my_rows;   // signal rows of (rank rR, slice j, this ring)
    __shared__ uint32_t *s_to_rows;         // signal rows of (rank down, slice j, this ring)
    __shared__ unsigned long long *s_stampR, *s_stampL;   // step stamps of ranks rR and rL, or null
    extern __shared__ __align__(16) unsigned char s_hand[];   // p.hand_bytes: the handed-over head
    if (threadIdx.x == 0) {
        s_epoch0 = ld_relaxed_gpu(&p.hdr->epoch);
        s_abort = 0;
        s_my_rows = p.sig + (((size_t)j * P + rR) * (size_t)p.rows + row_h) * P;
        s_to_rows = p.sig + (((size_t)j * P + down) * (size_t)p.rows + row_h) * P;
        // stamps keep k_ring's layout, one row per (half, rank, slice): row (h*P + r) * S + j
        const size_t hbase = BIDIR ? (size_t)hf * P : 0;
        const size_t rowR = (hbase + rR) * S + j, rowL = (hbase + rL) * S + j;
        s_stampR = (p.trace && (rowR + 1) * nsteps * 3 <= p.trace_words) ? p.trace + rowR * nsteps * 3 : nullptr;
        s_stampL = (p.trace && (rowL + 1) * nsteps * 3 <= p.trace_words) ? p.trace + rowL * nsteps * 3 : nullptr;
    }
    __syncthreads();
    if (p.stagger_groups > 1) {   // phase-shifted slice rings, as in k_ring
        const unsigned g = (unsigned)j % (unsigned)p.stagger_groups;
        if (g && threadIdx.x == 0) {
            const uint64_t t0 = global_timer_ns(), d = (uint64_t)g * p.stagger_ns;
            while (global_timer_ns() - t0 < d) __nanosleep(128);
        }
        __syncthreads();
    }
    const uint32_t E0 = s_epoch0;
    const uint32_t E = E0 + 1u;
    const size_t cs = p.chunk_stride;
    char *slotR = p.data + (size_t)rR * p.data_stride;
    char *slotL = p.data + (size_t)rL * p.data_stride;
    const char *slotU = p.data + (size_t)up * p.data_stride;
    const uint32_t sm = (uint32_t)__cvta_generic_to_shared(s_hand);
    constexpr size_t kGroup = 1024 / ES;            // elements of one 32-vector group
    const size_t hmax = (size_t)p.hand_bytes / ES;  // a multiple of kGroup
    uint32_t meet_round = 0;

    const size_t half = p.chunk / 2;
    const size_t range_lo = BIDIR ? (hf == 0 ? 0 : half) : 0;   // element range of this ring in every chunk
    const size_t range_n = BIDIR ? (hf == 0 ? half : p.chunk - half) : p.chunk;
    for (int q = 0; q < p.segments; ++q) {
        const size_t seg_lo = range_lo + slice_begin(range_n, q, p.segments);
        const size_t seg_n = range_lo + slice_begin(range_n, q + 1, p.segments) - seg_lo;
        const size_t lo = seg_lo + slice_begin(seg_n, j, S);
        const size_t n = seg_lo + slice_begin(seg_n, j + 1, S) - lo;
        const uint32_t V = E0 + 1u + (uint32_t)q;
        size_t h = n < hmax ? n : hmax;   // head elements handed over in shared memory
        h -= h % kGroup;
        const size_t hv = h * ES / 32;
        const size_t hb = h * ES;

        for (int g = 0; g < nsteps; ++g) {
            // Step stamps (thread 0, first segment): rank rL waits on no other
            // block, so its wait starts and ends when its step starts.
            if (threadIdx.x == 0 && s_stampL && q == 0) s_stampL[3 * g] = s_stampL[3 * g + 1] = global_timer_ns();
            const bool last = g == nsteps - 1;
            // ---- 1. rank rL, step g
            if (g < P - 1) {
                const int s = g;
                const int k = chunk_of(rL, s);
                const size_t off = ((size_t)k * cs + lo) * ES;
                const char *a = slotR + off;   // rR's output of step s-1 (s = 0: rR's input chunk)
                char *own = slotL + off;
                // the last reduce-scatter step stores the finished chunk k to its owner's out slot
                char *dst = (MODE != MODE_ALLREDUCE && s == P - 2) ? p.out + (size_t)k * p.out_stride + lo * ES : own;
                const bool drop = p.discard && s >= 1;
                if (p.discard && s < P - 2) {   // a partial the next block reads next step: keep it in L2
                    if (s == 0)
                        head_add<DT, T, false, false, true, kStEvictLast>(dst, sm, a, own, hv, false);
                    else
                        head_add<DT, T, true, false, true, kStEvictLast>(dst, sm, a, own, hv, false);
                    add_range<DT, T, kStEvictLast>(dst + hb, a + hb, own + hb, n - h, drop);
                } else if constexpr (MODE != MODE_ALLREDUCE) {   // the output chunk
                    if (s == 0)
                        head_add<DT, T, false, false, true, kStNormal>(dst, sm, a, own, hv, false);
                    else
                        head_add<DT, T, true, false, true, kStNormal>(dst, sm, a, own, hv, false);
                    add_range<DT, T, kStNormal>(dst + hb, a + hb, own + hb, n - h, drop);
                } else {   // the reduced chunk, read by the next block in the first all-gather step
                    if (s == 0)
                        head_add<DT, T, false, false, true, kPolReadNext>(dst, sm, a, own, hv, false);
                    else
                        head_add<DT, T, true, false, true, kPolReadNext>(dst, sm, a, own, hv, false);
                    add_range<DT, T, kPolReadNext>(dst + hb, a + hb, own + hb, n - h, drop);
                }
            } else {
                const int t = g - (P - 1);
                const int k = (rL - 1 - t + 2 * P) % P;
                const size_t off = ((size_t)k * cs + lo) * ES;
                if (last) {
                    head_copy<T, true, false, kStEvictFirst>(slotL + off, sm, slotR + off, hv);
                    copy_range<ES, T, kStEvictFirst>(slotL + off + hb, slotR + off + hb, n - h);
                } else {
                    head_copy<T, true, false, kPolReadNext>(slotL + off, sm, slotR + off, hv);
                    copy_range<ES, T, kPolReadNext>(slotL + off + hb, slotR + off + hb, n - h);
                }
            }
            // ---- 2. every thread's stores (and reads of the shared head) precede the notify
            __syncthreads();
            // (test hook: a skip aimed at either rank of the block skips the block's notify)
            if (g + 1 < nsteps && threadIdx.x == 0 && !((r0 == p.skip_rank || r1 == p.skip_rank) && g == p.skip_step))
                st_release_gpu(&s_to_rows[(size_t)(g + 1) * P + rL], V);
            if (threadIdx.x == 0 && q == 0) {
                const unsigned long long now = (s_stampR || s_stampL) ? global_timer_ns() : 0ull;
                if (s_stampL) s_stampL[3 * g + 2] = now;
                if (s_stampR) s_stampR[3 * g] = now;
            }
            // ---- 3. wait for rR's upstream neighbour, in the neighbouring block
            if (g > 0) {
                if (threadIdx.x == 0 && !wait_row(&s_my_rows[(size_t)g * P + up], V, E, p, rR, g, j, abort_word))
                    s_abort = 1;
                __syncthreads();
                if (s_abort) break;
            }
            if (threadIdx.x == 0 && s_stampR && q == 0) s_stampR[3 * g + 1] = global_timer_ns();
            // ---- 4. rank rR, step g
            if (g < P - 1) {
                const int s = g;
                const int k = chunk_of(rR, s);
                const size_t off = ((size_t)k * cs + lo) * ES;
                const char *a = slotU + off;
                char *own = slotR + off;
                const bool drop = p.discard && s >= 1;
                if (MODE != MODE_ALLREDUCE && s == P - 2) {   // the finished chunk: to its owner's output only
                    char *dst = p.out + (size_t)k * p.out_stride + lo * ES;
                    head_add<DT, T, false, false, true, kStNormal>(dst, sm, a, own, hv, drop);
                    add_range<DT, T, kStNormal>(dst + hb, a + hb, own + hb, n - h, drop);
                } else if (s == P - 2) {   // all-reduce: the reduced chunk to the slot, its head also to r1
                    head_add<DT, T, false, true, true, kPolNoReread>(own, sm, a, own, hv, drop);
                    add_range<DT, T, kPolReadNext>(own + hb, a + hb, own + hb, n - h, drop);
                } else {   // a partial: its head to r1 through shared memory only, the rest to the slot
                    head_add<DT, T, false, true, false, kStNormal>(own, sm, a, own, hv, drop);
                    if (p.discard)
                        add_range<DT, T, kStEvictLast>(own + hb, a + hb, own + hb, n - h, drop);
                    else
                        add_range<DT, T, kStNormal>(own + hb, a + hb, own + hb, n - h, drop);
                }
            } else {
                const int t = g - (P - 1);
                const int k = (rR - 1 - t + 2 * P) % P;
                const size_t off = ((size_t)k * cs + lo) * ES;
                if (last) {
                    head_copy<T, false, false, kStEvictFirst>(slotR + off, sm, slotU + off, hv);
                    copy_range<ES, T, kStEvictFirst>(slotR + off + hb, slotU + off + hb, n - h);
                } else {
                    head_copy<T, false, true, kPolNoReread>(slotR + off, sm, slotU + off, hv);
                    copy_range<ES, T, kPolReadNext>(slotR + off + hb, slotU + off + hb, n - h);
                }
            }
            __syncthreads();   // the shared head is complete before rank rL reads it
            if (threadIdx.x == 0 && s_stampR && q == 0) s_stampR[3 * g + 2] = global_timer_ns();
            if constexpr (SERIAL) {
                grid_meet(p, ++meet_round, E, abort_word, rR, g, j, &s_abort);
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
            p.hdr->pad[1] = 0;
            st_relaxed_gpu(&p.hdr->epoch, E0 + (uint32_t)p.segments);
        }
    }
}

// ------------------------------------------------------------ host launchers
template <int DT, bool SERIAL>
static const void *pair_fn_mode(int mode)
{
    return mode == MODE_ALLREDUCE       ? (const void *)k_ring_pair<DT, MODE_ALLREDUCE, SERIAL>
           : mode == MODE_RS_BIDIR      ? (const void *)k_ring_pair<DT, MODE_RS_BIDIR, SERIAL>
                                        : (const void *)k_ring_pair<DT, MODE_REDUCE_SCATTER, SERIAL>;
}
constexpr int kPairModes[3] = {MODE_ALLREDUCE, MODE_REDUCE_SCATTER, MODE_RS_BIDIR};

static const void *pair_fn(int dtype, int mode, bool serial)
{
    if (serial) {
        switch (dtype) {
        case 0: return pair_fn_mode<0, true>(mode);
        case 1: return pair_fn_mode<1, true>(mode);
        default: return pair_fn_mode<2, true>(mode);
        }
    }
    switch (dtype) {
    case 0: return pair_fn_mode<0, false>(mode);
    case 1: return pair_fn_mode<1, false>(mode);
    default: return pair_fn_mode<2, false>(mode);
    }
}

// Every instantiation may take hand_bytes of dynamic shared memory.
static cudaError_t pair_allow_smem(int hand_bytes)
{
    for (int dt = 0; dt < 3; ++dt)
        for (int mode = 0; mode < 6; ++mode) {
            const void *f = pair_fn(dt, kPairModes[mode % 3], mode >= 3);
            cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, hand_bytes);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t ring_pair_max_coresident(int dtype, int device, int hand_bytes, int *blocks)
{
    cudaError_t e = pair_allow_smem(hand_bytes);
    if (e != cudaSuccess) return e;
    int sms = 0, best = 1 << 30;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    for (int mode = 0; mode < 6; ++mode) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pair_fn(dtype, kPairModes[mode % 3], mode >= 3),
                                                          kPairThreads, (size_t)hand_bytes);
        if (e != cudaSuccess) return e;
        if (per_sm < best) best = per_sm;
    }
    *blocks = best * sms;
    return cudaSuccess;
}

cudaError_t launch_ring_pair(const RingParams &p, int dtype, cudaStream_t st)
{
    RingParams copy = p;
    if (copy.chunk_stride == 0) copy.chunk_stride = copy.chunk;
    void *args[] = {(void *)&copy};
    const unsigned blocks = (unsigned)(p.P / 2 * p.S) * (p.mode == MODE_RS_BIDIR ? 2u : 1u);
    return cudaLaunchCooperativeKernel(pair_fn(dtype, copy.mode, copy.debug_serial != 0), dim3(blocks),
                                       dim3((unsigned)kPairThreads), args, (size_t)copy.hand_bytes, st);
}

} // namespace rc
