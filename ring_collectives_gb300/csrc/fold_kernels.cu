// fold_kernels.cu -- single-pass all-reduces: every element position of all
// P slots is read once and written once (2*P*N*e bytes, the minimum), the
// per-element fold happening on chip.
//
// Two fold orders share the kernel:
//  * RING: the ring all-reduce's own result, R[k] = ((x_{k+1} + x_{k+2}) +
//    ...) + x_k for an element of chunk k ("全归约 3：Ring——每步大小恒定",
//    section "走读": the reduce-scatter rounds fold chunk k starting at rank
//    k+1 and ending at rank k).  Bit-identical to ring_allreduce; this is
//    the ring without its 2(P-1) passes over HBM.
//  * PSUM: the rotate-and-accumulate all-reduce of "Pallas TPU Distributed
//    Collectives 复习文档", section 3 (psum): rank r starts from 0 and adds the
//    block arriving from its left at each of P steps, x_{r-1}, x_{r-2}, ...,
//    x_r, so every rank folds in its own order.  On one GPU the rotation's hops
//    cost nothing: the block for step t of rank r is slot (r-1-t) mod P, read
//    from the tile already on chip.
//
// Register form (P <= 8, slots 32-byte aligned): each thread loads the same
// 32-byte vector of all P slots into registers (coalesced across the warp,
// evict-first), folds it with P fixed at compile time so every operand index
// is static, and stores the P results.  The only memory traffic is the P
// reads and P writes of each position.  Vectors that straddle a chunk
// boundary and the ragged tail are folded element by element.
//
// Shared-memory form (any P or alignment): a block stages a tile of TE
// positions of all P slots in shared memory, then computes each output and
// stores it.  Each position is independent, so both forms are in place.
#include <cstdlib>

#include "dev.cuh"
#include "internal.h"
#include "ringcoll.h"

namespace rc {

constexpr int kFoldThreads = 256;
constexpr int kFoldSmem = 32 * 1024;   // bytes of staged tile per block

template <int DT>
__device__ __forceinline__ uint32_t fold_add(uint32_t a, uint32_t b)
{
    if (DT == 0) return add_f32_bits(a, b);
    if (DT == 1) return add_bf16_bits((uint16_t)a, (uint16_t)b);
    return a + b;
}

template <int ES>
__device__ __forceinline__ uint32_t sm_get(const unsigned char *tile, size_t idx)
{
    if (ES == 2) return ((const uint16_t *)tile)[idx];
    return ((const uint32_t *)tile)[idx];
}

template <int ES>
__device__ __forceinline__ void st_elem(char *p, uint32_t v)
{
    if (ES == 2)
        st_u16(p, (uint16_t)v);
    else
        st_u32(p, v);
}

__device__ __forceinline__ uint4 ld_ef_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// ORDER 0 = RING, 1 = PSUM.
template <int DT, int ORDER>
__global__ void __launch_bounds__(kFoldThreads) k_fold(char *data, size_t stride, int P, size_t N, size_t chunk,
                                                       int te)
{
    constexpr int ES = DT == 1 ? 2 : 4;
    extern __shared__ __align__(16) unsigned char tile[];   // [P][te] elements
    const size_t tiles = (N + te - 1) / te;
    const bool vec = ((((uintptr_t)data) | stride) & 15u) == 0;
    for (size_t tix = blockIdx.x; tix < tiles; tix += gridDim.x) {
        const size_t i0 = tix * (size_t)te;
        const int len = (int)min((size_t)te, N - i0);
        // ---- stage [P][len] into shared memory
        if (vec) {
            const int vpr = len * ES / 16;   // whole 16-byte vectors per row
            for (int q = threadIdx.x; q < P * vpr; q += kFoldThreads) {
                const int r = q / vpr, v = q - r * vpr;
                const uint4 x = ld_ef_v4(data + (size_t)r * stride + i0 * ES + (size_t)v * 16);
                *(uint4 *)(tile + ((size_t)r * te) * ES + (size_t)v * 16) = x;
            }
            const int done = vpr * 16 / ES;
            for (int q = threadIdx.x; q < P * (len - done); q += kFoldThreads) {
                const int r = q / (len - done), e = done + q % (len - done);
                const char *src = data + (size_t)r * stride + (i0 + e) * ES;
                if (ES == 2)
                    ((uint16_t *)tile)[(size_t)r * te + e] = ld_cg_u16(src);
                else
                    ((uint32_t *)tile)[(size_t)r * te + e] = ld_cg_u32(src);
            }
        } else {
            for (int q = threadIdx.x; q < P * len; q += kFoldThreads) {
                const int r = q / len, e = q % len;
                const char *src = data + (size_t)r * stride + (i0 + e) * ES;
                if (ES == 2)
                    ((uint16_t *)tile)[(size_t)r * te + e] = ld_cg_u16(src);
                else
                    ((uint32_t *)tile)[(size_t)r * te + e] = ld_cg_u32(src);
            }
        }
        __syncthreads();
        // ---- fold and store: each thread handles VE consecutive positions
        // (one 16-byte shared-memory vector per source rank); the source rank
        // steps by +-1 with wrap-around instead of a modulo per term.
        constexpr int VE = 16 / ES;
        const int nv = (len + VE - 1) / VE;
        if (ORDER == 0) {
            for (int v = threadIdx.x; v < nv; v += kFoldThreads) {
                const int e0 = v * VE;
                const size_t i = i0 + e0;
                const int cnt = min(VE, len - e0);
                const size_t k0 = i / chunk, k1 = (i + cnt - 1) / chunk;
                if (k0 == k1 && cnt == VE) {
                    // whole vector in chunk k0: R = ((x_{k+1} + x_{k+2}) + ...) + x_k
                    int src = (int)((k0 + 1) % (size_t)P);
                    uint4 acc = *(const uint4 *)(tile + ((size_t)src * te + e0) * ES);
                    for (int jj = 2; jj <= P; ++jj) {
                        src = src + 1 == P ? 0 : src + 1;
                        acc = hop_add_v4<DT>(acc, *(const uint4 *)(tile + ((size_t)src * te + e0) * ES));
                    }
                    const bool gvec = vec; // rows 16-byte aligned: i*ES is, since e0 and i0 are VE-aligned
                    for (int r = 0; r < P; ++r) {
                        char *dst = data + (size_t)r * stride + i * ES;
                        if (gvec) {
                            st_v4(dst, acc);
                        } else {
                            const uint32_t w[4] = {acc.x, acc.y, acc.z, acc.w};
                            for (int q = 0; q < VE; ++q)
                                st_elem<ES>(dst + q * ES, ES == 2 ? (w[q >> 1] >> (16 * (q & 1))) & 0xFFFFu : w[q]);
                        }
                    }
                } else {
                    for (int q = 0; q < cnt; ++q) {
                        const size_t ii = i + q;
                        const int k = (int)(ii / chunk);
                        int src = k + 1 == P ? 0 : k + 1;
                        uint32_t acc = sm_get<ES>(tile, (size_t)src * te + e0 + q);
                        for (int jj = 2; jj <= P; ++jj) {
                            src = src + 1 == P ? 0 : src + 1;
                            acc = fold_add<DT>(acc, sm_get<ES>(tile, (size_t)src * te + e0 + q));
                        }
                        for (int r = 0; r < P; ++r) st_elem<ES>(data + (size_t)r * stride + ii * ES, acc);
                    }
                }
            }
        } else {
            for (int q2 = threadIdx.x; q2 < P * nv; q2 += kFoldThreads) {
                const int r = q2 / nv, v = q2 - r * nv;
                const int e0 = v * VE;
                const int cnt = min(VE, len - e0);
                int src = r == 0 ? P - 1 : r - 1;       // step 0 receives x_{r-1}
                char *dst = data + (size_t)r * stride + (i0 + e0) * ES;
                if (cnt == VE) {
                    uint4 acc = make_uint4(0, 0, 0, 0);  // +0.0 / bf16 +0 / int 0
                    for (int t = 0; t < P; ++t) {
                        acc = hop_add_v4<DT>(acc, *(const uint4 *)(tile + ((size_t)src * te + e0) * ES));
                        src = src == 0 ? P - 1 : src - 1;
                    }
                    if (vec) {
                        st_v4(dst, acc);
                    } else {
                        const uint32_t w[4] = {acc.x, acc.y, acc.z, acc.w};
                        for (int q = 0; q < VE; ++q)
                            st_elem<ES>(dst + q * ES, ES == 2 ? (w[q >> 1] >> (16 * (q & 1))) & 0xFFFFu : w[q]);
                    }
                } else {
                    for (int q = 0; q < cnt; ++q) {
                        int s2 = src;
                        uint32_t acc = 0;
                        for (int t = 0; t < P; ++t) {
                            acc = fold_add<DT>(acc, sm_get<ES>(tile, (size_t)s2 * te + e0 + q));
                            s2 = s2 == 0 ? P - 1 : s2 - 1;
                        }
                        st_elem<ES>(dst + q * ES, acc);
                    }
                }
            }
        }
        __syncthreads(); // the tile is reused by the next iteration
    }
}

// ------------------------------------------------------------ register form
constexpr int kFoldRegThreads = 256;

struct V32 {
    uint4 a, b;
};

template <int DT>
__device__ __forceinline__ V32 add32(const V32 &x, const V32 &y)
{
    return V32{hop_add_v4<DT>(x.a, y.a), hop_add_v4<DT>(x.b, y.b)};
}

// Ring order for chunk K: ((x_{K+1} + x_{K+2}) + ...) + x_K.
template <int DT, int PC, int K>
__device__ __forceinline__ V32 ring_fold(const V32 (&x)[PC])
{
    V32 acc = x[(K + 1) % PC];
#pragma unroll
    for (int jj = 2; jj <= PC; ++jj) acc = add32<DT>(acc, x[(K + jj) % PC]);
    return acc;
}

// Runtime chunk index -> the compile-time fold of that chunk.
template <int DT, int PC, int K = 0>
__device__ __forceinline__ V32 ring_fold_k(int k, const V32 (&x)[PC])
{
    if constexpr (K + 1 < PC) {
        if (k == K) return ring_fold<DT, PC, K>(x);
        return ring_fold_k<DT, PC, K + 1>(k, x);
    } else {
        return ring_fold<DT, PC, K>(x);
    }
}

// Position e of every slot, element by element (chunk-straddling vectors and
// the tail).
template <int DT, int ORDER>
__device__ void fold_elem(char *data, size_t stride, int P, size_t e, size_t chunk)
{
    constexpr int ES = DT == 1 ? 2 : 4;
    auto ld = [&](int r) -> uint32_t {
        const char *q = data + (size_t)r * stride + e * ES;
        return ES == 2 ? (uint32_t)ld_cg_u16(q) : ld_cg_u32(q);
    };
    if (ORDER == 0) {
        const int k = (int)(e / chunk);
        int src = k + 1 == P ? 0 : k + 1;
        uint32_t acc = ld(src);
        for (int jj = 2; jj <= P; ++jj) {
            src = src + 1 == P ? 0 : src + 1;
            acc = fold_add<DT>(acc, ld(src));
        }
        for (int r = 0; r < P; ++r) st_elem<ES>(data + (size_t)r * stride + e * ES, acc);
    } else {
        uint32_t out[8];
        for (int r = 0; r < P; ++r) {
            int src = r == 0 ? P - 1 : r - 1;
            uint32_t acc = 0;
            for (int t = 0; t < P; ++t) {
                acc = fold_add<DT>(acc, ld(src));
                src = src == 0 ? P - 1 : src - 1;
            }
            out[r] = acc;
        }
        for (int r = 0; r < P; ++r) st_elem<ES>(data + (size_t)r * stride + e * ES, out[r]);
    }
}

// ORDER 0 = RING, 1 = PSUM; PC = P.  data and stride are 32-byte aligned.
// Two blocks per SM (<= 128 registers), except the psum order at P >= 7,
// whose P live outputs need more registers than that.
template <int ORDER, int PC>
constexpr int fold_reg_min_blocks() { return (ORDER == 1 && PC >= 7) ? 1 : 2; }

template <int DT, int ORDER, int PC>
__global__ void __launch_bounds__(kFoldRegThreads, fold_reg_min_blocks<ORDER, PC>()) k_fold_reg(char *data, size_t stride, size_t N, size_t chunk)
{
    constexpr int ES = DT == 1 ? 2 : 4;
    constexpr int VE = 32 / ES;   // elements per 32-byte vector
    const size_t nvec = N / VE;
    const size_t step = (size_t)gridDim.x * kFoldRegThreads;
    for (size_t v = (size_t)blockIdx.x * kFoldRegThreads + threadIdx.x; v < nvec; v += step) {
        const size_t i = v * VE;
        const size_t off = i * ES;
        if (ORDER == 0) {
            const size_t k = i / chunk;
            if (i + VE > (k + 1) * chunk) {   // straddles chunks k and k+1
                for (int q = 0; q < VE; ++q) fold_elem<DT, 0>(data, stride, PC, i + q, chunk);
                continue;
            }
            V32 x[PC];
#pragma unroll
            for (int r = 0; r < PC; ++r) ld8_ef(data + (size_t)r * stride + off, x[r].a, x[r].b);
            const V32 acc = ring_fold_k<DT, PC>((int)k, x);
#pragma unroll
            for (int r = 0; r < PC; ++r) st8<kStEvictFirst>(data + (size_t)r * stride + off, acc.a, acc.b);
        } else {
            V32 x[PC];
#pragma unroll
            for (int r = 0; r < PC; ++r) ld8_ef(data + (size_t)r * stride + off, x[r].a, x[r].b);
            // rank r: +0, then x_{r-1}, x_{r-2}, ..., x_r
#pragma unroll
            for (int r = 0; r < PC; ++r) {
                V32 acc{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
#pragma unroll
                for (int t = 0; t < PC; ++t) acc = add32<DT>(acc, x[(r - 1 - t + 2 * PC) % PC]);
                st8<kStEvictFirst>(data + (size_t)r * stride + off, acc.a, acc.b);
            }
        }
    }
    // ragged tail: N % VE positions
    const size_t tail0 = nvec * VE;
    for (size_t e = tail0 + (size_t)blockIdx.x * kFoldRegThreads + threadIdx.x; e < N; e += step)
        fold_elem<DT, ORDER>(data, stride, PC, e, chunk);
}

template <int DT, int ORDER>
static const void *fold_reg_fn(int P)
{
    switch (P) {
    case 2: return (const void *)k_fold_reg<DT, ORDER, 2>;
    case 3: return (const void *)k_fold_reg<DT, ORDER, 3>;
    case 4: return (const void *)k_fold_reg<DT, ORDER, 4>;
    case 5: return (const void *)k_fold_reg<DT, ORDER, 5>;
    case 6: return (const void *)k_fold_reg<DT, ORDER, 6>;
    case 7: return (const void *)k_fold_reg<DT, ORDER, 7>;
    case 8: return (const void *)k_fold_reg<DT, ORDER, 8>;
    default: return nullptr;
    }
}

static const void *fold_reg_any(int dtype, int order, int P)
{
    if (order == 0) return dtype == 0 ? fold_reg_fn<0, 0>(P) : dtype == 1 ? fold_reg_fn<1, 0>(P) : fold_reg_fn<2, 0>(P);
    return dtype == 0 ? fold_reg_fn<0, 1>(P) : dtype == 1 ? fold_reg_fn<1, 1>(P) : fold_reg_fn<2, 1>(P);
}

// Knob, read once: RC_FOLD_BLOCKS = blocks per SM of the register fold
// (unset or malformed: the rule in launch_fold).
static int fold_blocks_setting()
{
    static const int v = [] {
        const char *e = getenv("RC_FOLD_BLOCKS");
        if (!e || !*e) return 0;
        char *end = nullptr;
        const long x = strtol(e, &end, 10);
        return (end && *end == 0 && x >= 1 && x <= 16) ? (int)x : 0;
    }();
    return v;
}

cudaError_t launch_fold(char *data, size_t stride, int P, size_t N, size_t chunk, int dtype, int order, int sm_count,
                        cudaStream_t st)
{
    const int es = dtype == 1 ? 2 : 4;
    const void *rf = ((((uintptr_t)data) | stride) & 31u) == 0 ? fold_reg_any(dtype, order, P) : nullptr;
    if (rf) {
        // 256-thread blocks over a grid-stride loop: as many per SM as fit, but
        // no more than keep ~64 KiB of loads in flight per SM (each thread holds
        // P vectors of 32 bytes: max(1, 8/P) blocks).  Measured on GB300 at P=8
        // x 64 MiB fp32, ring order: 2 blocks per SM 0.1679 ms, 1 block
        // 0.1637 ms (the psum order, whose registers allow 1 block, 0.1636).
        static int per_sm[3][2][9] = {};
        int &occ = per_sm[dtype][order][P];
        if (occ == 0) {
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rf, kFoldRegThreads, 0);
            if (e != cudaSuccess) return e;
            const int cap = fold_blocks_setting() > 0 ? fold_blocks_setting() : (8 / P > 1 ? 8 / P : 1);
            if (occ > cap) occ = cap;
            if (occ < 1) occ = 1;
        }
        const size_t vecs = N * es / 32 + 1;
        size_t grid = (size_t)sm_count * occ;
        const size_t need = (vecs + kFoldRegThreads - 1) / kFoldRegThreads;
        if (grid > need) grid = need;
        if (grid < 1) grid = 1;
        void *args[] = {(void *)&data, (void *)&stride, (void *)&N, (void *)&chunk};
        return cudaLaunchKernel(rf, dim3((unsigned)grid), dim3(kFoldRegThreads), args, 0, st);
    }
    int te = kFoldSmem / (P * es);
    te -= te % 64;
    if (te < 64) te = 64;
    const size_t smem = (size_t)P * te * es;
    const size_t tiles = (N + te - 1) / te;
    size_t grid = (size_t)sm_count * 6;
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    void (*fn)(char *, size_t, int, size_t, size_t, int);
    if (order == 0)
        fn = dtype == 0 ? k_fold<0, 0> : dtype == 1 ? k_fold<1, 0> : k_fold<2, 0>;
    else
        fn = dtype == 0 ? k_fold<0, 1> : dtype == 1 ? k_fold<1, 1> : k_fold<2, 1>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    fn<<<(unsigned)grid, kFoldThreads, smem, st>>>(data, stride, P, N, chunk, te);
    return cudaGetLastError();
}

} // namespace rc
