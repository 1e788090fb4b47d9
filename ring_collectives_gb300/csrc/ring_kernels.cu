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
// Why no extra guard against overwriting data a neighbour still reads: rank
// r reads its left neighbour's chunk (r-s-2) in round s; the left neighbour
// rewrites that chunk only in all-gather round s (global step P-1+s), and
// reaching that step needs a chain of P-1 notifies around the ring that ends
// with rank r's notify of step s, issued after rank r's loads of step s.
#include "internal.h"
#include "dev.cuh"
#include "ringcoll.h"

namespace rc {

constexpr int kUnroll = 4; // 16-byte vectors in flight per thread and operand

// First element of slice j of a chunk of c elements (slices are granule-aligned).
__device__ __forceinline__ size_t slice_begin(size_t c, int j, int S)
{
    if (j >= S) return c;
    const size_t b = (c * (size_t)j) / (size_t)S;
    return b - (b % kSliceGranule);
}

// ------------------------------------------------------------ block-wide streams
// dst[i] = a[i] (+) b[i] over nvec 16-byte vectors, strided over the block.
// T is the block size (a compile-time constant, so the unrolled offsets are
// immediates and only the three running pointers stay live).
template <int DT, int T>
__device__ __forceinline__ void add_vec(char *dst, const char *a, const char *b, size_t nvec)
{
    size_t v = threadIdx.x;
    const char *pa = a + v * 16, *pb = b + v * 16;
    char *pd = dst + v * 16;
    for (; v + (kUnroll - 1) * T < nvec; v += kUnroll * T) {
        uint4 x[kUnroll], y[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            x[u] = ld_cg_v4(pa + u * T * 16);
            y[u] = ld_cg_v4(pb + u * T * 16);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) st_v4(pd + u * T * 16, hop_add_v4<DT>(x[u], y[u]));
        pa += kUnroll * T * 16;
        pb += kUnroll * T * 16;
        pd += kUnroll * T * 16;
    }
    for (; v < nvec; v += T, pa += T * 16, pb += T * 16, pd += T * 16)
        st_v4(pd, hop_add_v4<DT>(ld_cg_v4(pa), ld_cg_v4(pb)));
}

template <int T>
__device__ __forceinline__ void copy_vec(char *dst, const char *src, size_t nvec)
{
    size_t v = threadIdx.x;
    const char *ps = src + v * 16;
    char *pd = dst + v * 16;
    for (; v + (kUnroll - 1) * T < nvec; v += kUnroll * T) {
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) x[u] = ld_cg_v4(ps + u * T * 16);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) st_v4(pd + u * T * 16, x[u]);
        ps += kUnroll * T * 16;
        pd += kUnroll * T * 16;
    }
    for (; v < nvec; v += T, ps += T * 16, pd += T * 16) st_v4(pd, ld_cg_v4(ps));
}

template <int DT>
__device__ __forceinline__ void add_scalar(char *dst, const char *a, const char *b, size_t n)
{
    for (size_t i = threadIdx.x; i < n; i += blockDim.x) {
        if (DT == 1)
            st_u16(dst + 2 * i, add_bf16_bits(ld_cg_u16(a + 2 * i), ld_cg_u16(b + 2 * i)));
        else if (DT == 0)
            st_u32(dst + 4 * i, add_f32_bits(ld_cg_u32(a + 4 * i), ld_cg_u32(b + 4 * i)));
        else
            st_u32(dst + 4 * i, ld_cg_u32(a + 4 * i) + ld_cg_u32(b + 4 * i));
    }
}

template <int ES>
__device__ __forceinline__ void copy_scalar(char *dst, const char *src, size_t n)
{
    for (size_t i = threadIdx.x; i < n; i += blockDim.x) {
        if (ES == 2)
            st_u16(dst + 2 * i, ld_cg_u16(src + 2 * i));
        else
            st_u32(dst + 4 * i, ld_cg_u32(src + 4 * i));
    }
}

// n elements; vec: all three pointers are 16-byte aligned.
template <int DT, int T>
__device__ __forceinline__ void add_range(char *dst, const char *a, const char *b, size_t n, bool vec)
{
    constexpr size_t ES = DT == 1 ? 2 : 4;
    size_t head = 0;
    if (vec) {
        const size_t nvec = (n * ES) / 16;
        add_vec<DT, T>(dst, a, b, nvec);
        head = nvec * 16 / ES;
    }
    add_scalar<DT>(dst + head * ES, a + head * ES, b + head * ES, n - head);
}

template <int ES, int T>
__device__ __forceinline__ void copy_range(char *dst, const char *src, size_t n, bool vec)
{
    size_t head = 0;
    if (vec) {
        const size_t nvec = (n * ES) / 16;
        copy_vec<T>(dst, src, nvec);
        head = nvec * 16 / ES;
    }
    copy_scalar<ES>(dst + head * ES, src + head * ES, n - head);
}

// ------------------------------------------------------------ bounded wait
// Spins (one thread) until *flag reaches epoch E.  Gives up when the launch
// has already failed elsewhere, or after timeout_ns: the first block to time
// out records RC_ERR_TIMEOUT with its rank/step/slice in the header.  Never
// traps; the caller returns cleanly and the host reads the status.
__device__ bool wait_row(const uint32_t *flag, uint32_t E, const RingParams &p, int r, int g, int j,
                         uint32_t *abort_word)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (epoch_reached(ld_acquire_gpu(flag), E)) return true;
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

// ------------------------------------------------------------ the step engine
template <int DT>
__global__ void __launch_bounds__(kRingThreads, 2) k_ring(const RingParams p)
{
    constexpr size_t ES = DT == 1 ? 2 : 4;
    const int P = p.P, S = p.S;
    const int r = (int)(blockIdx.x / (unsigned)S), j = (int)(blockIdx.x % (unsigned)S);
    const int left = (r - 1 + P) % P, right = (r + 1) % P;
    // The abort word is the header's pad[0]: a launch that gives up stores its epoch there.
    uint32_t *abort_word = &p.hdr->pad[0];

    __shared__ uint32_t s_epoch;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        s_epoch = ld_relaxed_gpu(&p.hdr->epoch) + 1u;
        s_abort = 0;
    }
    __syncthreads();
    const uint32_t E = s_epoch;

    const size_t c = p.chunk;
    const size_t lo = slice_begin(c, j, S), n = slice_begin(c, j + 1, S) - lo;
    const bool vec = p.vec_ok != 0;
    const uint32_t *my_rows = p.sig + ((size_t)j * P + r) * (size_t)p.rows * P;   // [rows][P]
    uint32_t *right_rows = p.sig + ((size_t)j * P + right) * (size_t)p.rows * P;
    char *my_slot = p.data + (size_t)r * p.data_stride;
    const char *left_slot = p.data + (size_t)left * p.data_stride;

    int nsteps;
    if (p.mode == MODE_ALL_GATHER) {
        nsteps = P - 1;
        // Prologue: the own shard goes to chunk r of the own output slot,
        // then row 0 of the right neighbour says it may be read.
        copy_range<ES, kRingThreads>(my_slot + ((size_t)r * c + lo) * ES, p.in + (size_t)r * p.in_stride + lo * ES, n, vec);
        __syncthreads();
        if (threadIdx.x == 0 && nsteps > 0) st_release_gpu(&right_rows[(size_t)0 * P + r], E);
    } else {
        nsteps = p.mode == MODE_ALLREDUCE ? 2 * (P - 1) : P - 1;
    }

    for (int g = 0; g < nsteps; ++g) {
        if (g > 0 || p.mode == MODE_ALL_GATHER) {
            if (threadIdx.x == 0 && !wait_row(&my_rows[(size_t)g * P + left], E, p, r, g, j, abort_word))
                s_abort = 1;
            __syncthreads();
            if (s_abort) break;
        }
        if (p.mode == MODE_ALL_GATHER) {
            const int k = (r - 1 - g + P) % P;
            const size_t off = ((size_t)k * c + lo) * ES;
            copy_range<ES, kRingThreads>(my_slot + off, left_slot + off, n, vec);
        } else if (g < P - 1) {
            const int s = g;
            const int k = (r - s - 2 + P) % P; // recv_add_idx == left_send_idx
            const size_t off = ((size_t)k * c + lo) * ES;
            char *own = my_slot + off;
            char *dst = (p.mode == MODE_REDUCE_SCATTER && s == P - 2)
                            ? p.out + (size_t)r * p.out_stride + lo * ES
                            : own;
            add_range<DT, kRingThreads>(dst, left_slot + off, own, n, vec);
        } else {
            const int t = g - (P - 1);
            const int k = (r - 1 - t + P) % P;
            const size_t off = ((size_t)k * c + lo) * ES;
            copy_range<ES, kRingThreads>(my_slot + off, left_slot + off, n, vec);
        }
        if (g + 1 < nsteps) {
            __syncthreads(); // every thread's stores of this step precede the release below
            if (threadIdx.x == 0 && !(r == p.skip_rank && g == p.skip_step))
                st_release_gpu(&right_rows[(size_t)(g + 1) * P + r], E);
        }
    }

    // Epilogue: the last block to finish publishes the new epoch.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&p.hdr->done, 1u);
        if (prev == gridDim.x - 1) {
            p.hdr->done = 0;
            st_relaxed_gpu(&p.hdr->epoch, E);
        }
    }
}

// ------------------------------------------------------------ right shift
// dst_r = src_{(r-1+P)%P}: blockIdx.y is the destination rank, blocks along x
// split the slot into contiguous pieces.
template <int ES>
__global__ void __launch_bounds__(256) k_ppermute(const char *src, size_t ss, char *dst, size_t ds, int P,
                                                  size_t n, int vec_ok)
{
    const int r = blockIdx.y;
    const int left = (r - 1 + P) % P;
    const char *s = src + (size_t)left * ss;
    char *d = dst + (size_t)r * ds;
    if (vec_ok) {
        const size_t nvec = n * ES / 16;
        const size_t per = (nvec + gridDim.x - 1) / gridDim.x;
        const size_t b0 = per * blockIdx.x, b1 = min(nvec, b0 + per);
        if (b0 < b1) copy_vec<256>(d + b0 * 16, s + b0 * 16, b1 - b0);
        if (blockIdx.x == 0) {
            const size_t head = nvec * 16 / ES;
            copy_scalar<ES>(d + head * ES, s + head * ES, n - head);
        }
    } else {
        const size_t per = (n + gridDim.x - 1) / gridDim.x;
        const size_t b0 = per * blockIdx.x, b1 = min(n, b0 + per);
        if (b0 < b1) copy_scalar<ES>(d + b0 * ES, s + b0 * ES, b1 - b0);
    }
}

// ------------------------------------------------------------ host launchers
static const void *ring_fn(int dtype)
{
    switch (dtype) {
    case 0: return (const void *)k_ring<0>;
    case 1: return (const void *)k_ring<1>;
    default: return (const void *)k_ring<2>;
    }
}

cudaError_t ring_max_coresident(int dtype, int threads, int device, int *blocks)
{
    int per_sm = 0, sms = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ring_fn(dtype), threads, 0);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    *blocks = per_sm * sms;
    return cudaSuccess;
}

cudaError_t launch_ring(const RingParams &p, int dtype, int threads, cudaStream_t st)
{
    RingParams copy = p;
    void *args[] = {(void *)&copy};
    return cudaLaunchCooperativeKernel(ring_fn(dtype), dim3((unsigned)(p.P * p.S)), dim3((unsigned)threads),
                                       args, 0, st);
}

cudaError_t launch_ppermute(const char *src, size_t src_stride, char *dst, size_t dst_stride, int P, size_t n,
                            int esize, int vec_ok, int sm_count, cudaStream_t st)
{
    // About four blocks per SM in total, at least one per rank.
    const size_t bytes = n * (size_t)esize;
    unsigned bx = (unsigned)((4 * (size_t)sm_count + P - 1) / P);
    const size_t max_bx = (bytes + 16383) / 16384; // no block below ~16 KiB
    if (bx > max_bx) bx = (unsigned)max_bx;
    if (bx < 1) bx = 1;
    dim3 grid(bx, (unsigned)P);
    if (esize == 2)
        k_ppermute<2><<<grid, 256, 0, st>>>(src, src_stride, dst, dst_stride, P, n, vec_ok);
    else
        k_ppermute<4><<<grid, 256, 0, st>>>(src, src_stride, dst, dst_stride, P, n, vec_ok);
    return cudaGetLastError();
}

} // namespace rc
