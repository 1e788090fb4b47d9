// ring_common.cuh -- device building blocks shared by the ring step engines
// (k_ring in ring_kernels.cu, one logical rank per thread block, and k_ring_pair
// in ring_pair.cu, two ranks per thread block): slice bounds, the block-wide
// streaming add and copy loops, the bounded wait on a signal row and the
// barrier-injection debug meet.
#pragma once
#include "internal.h"
#include "dev.cuh"
#include "ringcoll.h"

namespace rc {

// First element of slice j of a chunk of c elements (slices are granule-aligned).
__device__ __forceinline__ size_t slice_begin(size_t c, int j, int S)
{
    if (j >= S) return c;
    const size_t b = (c * (size_t)j) / (size_t)S;
    return b - (b % kSliceGranule);
}

// ------------------------------------------------------------ block-wide streams
// Bodies move 32-byte vectors strided over the T threads of the block (T is a
// compile-time constant, so the unrolled offsets are immediates); each thread
// keeps 2 (add) or 4 (copy) vectors per operand in flight.  The last partial
// round issues all of its (predicated) loads before its stores, so short
// ranges do not pay one memory latency per vector.

// dst[i] = a[i] (+) b[i] over n32 32-byte vectors.  The unrolled loop is
// warp-uniform (every lane runs the same iterations).  With `discard`, each warp
// drops the L2 lines of `a` it has just consumed (when `discard` is set): after __syncwarp every lane's
// loads have returned (its store used them), so lane l discards line l of the
// warp's two 1 KiB pieces.  Only done when `a` is 128-byte aligned, so every
// discarded line lies wholly inside this warp's piece of the range.
// TAIL_DROP: the last partial round drops its whole lines of `a` too (measured
// on GB300: faster in the all-reduces and in the two-rank reduce-scatter,
// slower in the one-rank-per-block reduce-scatters).
template <int DT, int T, int POL, bool TAIL_DROP = true>
__device__ __forceinline__ void add_vec32(char *dst, const char *a, const char *b, size_t n32, bool discard)
{
    constexpr int U = RC_RING_ADD_U;
    const size_t lane = threadIdx.x & 31u;
    size_t vw = threadIdx.x - lane; // first vector of this warp
    const bool dline = discard && (((uintptr_t)a & 127u) == 0);
    for (; vw + 31 + (U - 1) * T < n32; vw += U * T) {
        const size_t v = vw + lane;
        uint4 x0[U], x1[U], y0[U], y1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            ld8_ef(a + (v + u * T) * 32, x0[u], x1[u]);
            ld8_ef(b + (v + u * T) * 32, y0[u], y1[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            st8<POL>(dst + (v + u * T) * 32, hop_add_v4<DT>(x0[u], y0[u]), hop_add_v4<DT>(x1[u], y1[u]));
        if (dline) {
            __syncwarp();
            if (lane < 8 * U) discard_l2_line(a + (vw + (lane >> 3) * T) * 32 + (lane & 7) * 128);
        }
    }
    if (vw < n32) {   // at most one partial round is left for this warp
        const size_t v = vw + lane;
        if (v < n32) {
            uint4 x0[U] = {}, x1[U] = {}, y0[U] = {}, y1[U] = {};
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t ok = v + u * T < n32;
                ld8_ef_if(a + (v + u * T) * 32, ok, x0[u], x1[u]);
                ld8_ef_if(b + (v + u * T) * 32, ok, y0[u], y1[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v + u * T < n32)
                    st8<POL>(dst + (v + u * T) * 32, hop_add_v4<DT>(x0[u], y0[u]), hop_add_v4<DT>(x1[u], y1[u]));
        }
        if (TAIL_DROP && dline) {   // only lines that lie wholly inside the range
            __syncwarp();
            const size_t first = vw + (lane >> 3) * T + (lane & 7) * 4;
            if (lane < 8 * U && first + 4 <= n32) discard_l2_line(a + first * 32);
        }
    }
}

template <int T, int POL>
__device__ __forceinline__ void copy_vec32(char *dst, const char *src, size_t n32)
{
    constexpr int U = 4;
    size_t v = threadIdx.x;
    const char *ps = src + v * 32;
    char *pd = dst + v * 32;
    for (; v + (U - 1) * T < n32; v += U * T) {
        uint4 x0[U], x1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) ld8_ef(ps + u * T * 32, x0[u], x1[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) st8<POL>(pd + u * T * 32, x0[u], x1[u]);
        ps += U * T * 32;
        pd += U * T * 32;
    }
    if (v < n32) {   // at most one partial round is left for this thread
        uint4 x0[U] = {}, x1[U] = {};
#pragma unroll
        for (int u = 0; u < U; ++u) ld8_ef_if(ps + u * T * 32, v + u * T < n32, x0[u], x1[u]);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + u * T < n32) st8<POL>(pd + u * T * 32, x0[u], x1[u]);
    }
}

template <int DT, int T>
__device__ __forceinline__ void add_scalar(char *dst, const char *a, const char *b, size_t n)
{
    for (size_t i = threadIdx.x; i < n; i += T) {
        if (DT == 1)
            st_u16(dst + 2 * i, add_bf16_bits(ld_cg_u16(a + 2 * i), ld_cg_u16(b + 2 * i)));
        else if (DT == 0)
            st_u32(dst + 4 * i, add_f32_bits(ld_cg_u32(a + 4 * i), ld_cg_u32(b + 4 * i)));
        else
            st_u32(dst + 4 * i, ld_cg_u32(a + 4 * i) + ld_cg_u32(b + 4 * i));
    }
}

template <int ES, int T>
__device__ __forceinline__ void copy_scalar(char *dst, const char *src, size_t n)
{
    for (size_t i = threadIdx.x; i < n; i += T) {
        if (ES == 2)
            st_u16(dst + 2 * i, ld_cg_u16(src + 2 * i));
        else
            st_u32(dst + 4 * i, ld_cg_u32(src + 4 * i));
    }
}

// Elements before the first 32-byte boundary of dst (all pointers must share
// dst's offset modulo 32 for the vector body to apply; otherwise the whole
// range is element-wise).
template <int ES>
__device__ __forceinline__ size_t vec_head(const void *dst, size_t n)
{
    const size_t mis = (uintptr_t)dst & 31u;
    const size_t h = mis ? (32 - mis) / ES : 0;
    return h < n ? h : n;
}

// dst[i] = a[i] (+) b[i], i < n.  discard: a's data is dead after this read
// (see add_vec32).
template <int DT, int T, int POL, bool TAIL_DROP = true>
__device__ __forceinline__ void add_range(char *dst, const char *a, const char *b, size_t n, bool discard)
{
    constexpr size_t ES = DT == 1 ? 2 : 4;
    const bool same = ((((uintptr_t)dst ^ (uintptr_t)a) | ((uintptr_t)dst ^ (uintptr_t)b)) & 31u) == 0;
    if (!same) {
        add_scalar<DT, T>(dst, a, b, n);
        return;
    }
    const size_t h = vec_head<ES>(dst, n);
    add_scalar<DT, T>(dst, a, b, h);
    const size_t n32 = (n - h) * ES / 32;
    add_vec32<DT, T, POL, TAIL_DROP>(dst + h * ES, a + h * ES, b + h * ES, n32, discard);
    const size_t done = h + n32 * 32 / ES;
    add_scalar<DT, T>(dst + done * ES, a + done * ES, b + done * ES, n - done);
}

template <int ES, int T, int POL>
__device__ __forceinline__ void copy_range(char *dst, const char *src, size_t n)
{
    if ((((uintptr_t)dst ^ (uintptr_t)src) & 31u) != 0) {
        copy_scalar<ES, T>(dst, src, n);
        return;
    }
    const size_t h = vec_head<ES>(dst, n);
    copy_scalar<ES, T>(dst, src, h);
    const size_t n32 = (n - h) * ES / 32;
    copy_vec32<T, POL>(dst + h * ES, src + h * ES, n32);
    const size_t done = h + n32 * 32 / ES;
    copy_scalar<ES, T>(dst + done * ES, src + done * ES, n - done);
}

// ------------------------------------------------------------ bounded wait
// Spins (one thread) until *flag reaches value V.  Gives up when the launch
// has already failed elsewhere, or after timeout_ns: the first block to time
// out records RC_ERR_TIMEOUT with its rank/step/slice in the header.  Never
// traps; the caller returns cleanly and the host reads the status.
__device__ inline bool wait_row(const uint32_t *flag, uint32_t V, uint32_t E, const RingParams &p, int r, int g, int j,
                         uint32_t *abort_word)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (epoch_reached(ld_acquire_gpu(flag), V)) return true;
        if ((it & 31u) == 31u) {
            if (ld_relaxed_gpu(abort_word) == E) return false;
            const uint64_t now = global_timer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > p.timeout_ns) {
                if (atomicCAS(&p.hdr->status, 0u, (unsigned)RC_ERR_TIMEOUT) == 0u) {
                    p.hdr->err_rank = (uint32_t)r;
                    p.hdr->err_step = (uint32_t)g;
                    p.hdr->err_slice = (uint32_t)j;
                }
                st_relaxed_gpu(abort_word, E);
                return false;
            }
        }
        __nanosleep(20);
    }
}

// ------------------------------------------------------------ debug grid barrier
// RC_DEBUG_SERIAL: after every step, all blocks of the launch meet.  Thread 0
// adds one arrival to a launch-wide counter (the header's pad[1], zero at the
// start of every launch: the last block to finish resets it) and waits,
// bounded like every other wait, until round * gridDim.x blocks have arrived.
__device__ inline void grid_meet(const RingParams &p, uint32_t round, uint32_t E, uint32_t *abort_word, int r, int g, int j,
                          int *abort_flag)
{
    __syncthreads();
    if (threadIdx.x == 0 && !*abort_flag) {
        uint32_t *ctr = &p.hdr->pad[1];
        __threadfence();
        atomicAdd(ctr, 1u);
        const uint32_t goal = round * gridDim.x;
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
            if ((int32_t)(ld_acquire_gpu(ctr) - goal) >= 0) break;
            if ((it & 31u) == 31u) {
                if (ld_relaxed_gpu(abort_word) == E) {
                    *abort_flag = 1;
                    break;
                }
                const uint64_t now = global_timer_ns();
                if (t0 == 0) {
                    t0 = now;
                } else if (now - t0 > p.timeout_ns) {
                    if (atomicCAS(&p.hdr->status, 0u, (unsigned)RC_ERR_TIMEOUT) == 0u) {
                        p.hdr->err_rank = (uint32_t)r;
                        p.hdr->err_step = (uint32_t)g;
                        p.hdr->err_slice = (uint32_t)j;
                    }
                    st_relaxed_gpu(abort_word, E);
                    *abort_flag = 1;
                    break;
                }
            }
            __nanosleep(32);
        }
    }
    __syncthreads();
}

} // namespace rc
