// dev.cuh -- device primitives of the ring kernels: release/acquire signal
// words, a bounded spin-wait, 16-byte vector loads/stores and the per-element
// hop add.  All inline PTX here is hand-written.
#pragma once
#include <stdint.h>
#include <cuda_runtime.h>

namespace rc {

// ------------------------------------------------------------ signal words
// A notify is a release store of the epoch value: every write the CTA made
// before it (ordered by the preceding __syncthreads) becomes visible to a
// thread that observes the value with an acquire load.  The Triton-distributed
// semantics page calls the pair notify / wait, and its consume_token is what
// the acquire (plus the "memory" clobber) gives here: no load of the signalled
// data can be hoisted above the wait.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Epoch comparison that survives 32-bit wrap-around: v has reached E.
__device__ __forceinline__ bool epoch_reached(uint32_t v, uint32_t E) { return (int32_t)(v - E) >= 0; }

// ------------------------------------------------------------ data movement
// Loads of slot data go through L2 only (.cg): the data was written by other
// thread blocks inside the same kernel, so the non-coherent read-only path
// must not be used, and L1 holds nothing worth keeping for a stream.
__device__ __forceinline__ uint4 ld_cg_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_cg_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint16_t ld_cg_u16(const void *p)
{
    uint16_t v;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_u32(void *p, uint32_t v)
{
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_u16(void *p, uint16_t v)
{
    asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

// 32-byte vectors (sm_100+ 256-bit global accesses).  Ring loads are the last
// use of their data on this step, so they carry L1::no_allocate and
// L2::evict_first: the just-written partials and chunks the neighbours read
// next keep their L2 lines instead.  Stores use the default policy, except the
// last all-gather step, whose output no one reads again (evict_first).
__device__ __forceinline__ void ld8_ef(const void *p, uint4 &a, uint4 &b)
{
    asm volatile("ld.global.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p)
                 : "memory");
}

// ld8_ef issued only when `valid` is non-zero (a PTX predicate); otherwise a
// and b are left as they were.
__device__ __forceinline__ void ld8_ef_if(const void *p, uint32_t valid, uint4 &a, uint4 &b)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %9, 0;\n\t"
                 "@q ld.global.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t}"
                 : "+r"(a.x), "+r"(a.y), "+r"(a.z), "+r"(a.w), "+r"(b.x), "+r"(b.y), "+r"(b.z), "+r"(b.w)
                 : "l"(p), "r"(valid)
                 : "memory");
}

// Store policies: kStNormal (output read by a neighbour next step), kStEvictFirst
// (nothing reads it again in this launch), kStEvictLast (a reduce-scatter
// partial: it must survive in L2 until the right neighbour reads it, which then
// drops it without write-back).
enum { kStNormal = 0, kStEvictFirst = 1, kStEvictLast = 2 };

template <int POL>
__device__ __forceinline__ void st8(void *p, const uint4 &a, const uint4 &b)
{
    if (POL == kStEvictFirst)
        asm volatile("st.global.L1::no_allocate.L2::evict_first.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                     "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                     : "memory");
    else if (POL == kStEvictLast)
        asm volatile("st.global.L1::no_allocate.L2::evict_last.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                     "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                     : "memory");
    else
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
                     "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                     : "memory");
}

// Drops one 128-byte L2 line without writing it back; the memory behind it is
// undefined afterwards, so only lines whose data is dead may be discarded.
// Fetch the 128-byte line at p into L2 (no registers, no completion wait).
__device__ __forceinline__ void prefetch_l2_line(const void *p)
{
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void discard_l2_line(const void *p)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// ------------------------------------------------------------ hop add
// Element types: 0 = f32, 1 = bf16, 2 = i32.
// f32: IEEE binary32 add, round to nearest even, subnormals kept (the library
//      is built without fast math / flush-to-zero).
// bf16: both operands widened to binary32 (exact), added in binary32, the sum
//      rounded to bf16 to nearest even.  Computed as one add.rn.bf16x2 (the
//      exact sum rounded once to bf16), which gives the same bits for every
//      pair of bf16 operands: whenever the binary32 sum is inexact, the
//      exponents differ by more than 16, the smaller operand lies below a
//      quarter of the larger's bf16 spacing, and both forms return the
//      larger operand.  Compared on GB300 for all 2^32 operand pairs: equal
//      except NaN payloads (both results are NaN for the same pairs).
// i32: two's-complement wrapping add.
__device__ __forceinline__ uint32_t add_f32_bits(uint32_t a, uint32_t b)
{
    return __float_as_uint(__fadd_rn(__uint_as_float(a), __uint_as_float(b)));
}

// Two packed bf16 (low half = element 0) -> two packed bf16 sums.
__device__ __forceinline__ uint32_t add_bf16x2_bits(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint16_t add_bf16_bits(uint16_t a, uint16_t b)
{
    return (uint16_t)(add_bf16x2_bits((uint32_t)a, (uint32_t)b) & 0xFFFFu);
}

template <int DT>
__device__ __forceinline__ uint4 hop_add_v4(uint4 a, uint4 b)
{
    uint4 r;
    if (DT == 0) {
        r.x = add_f32_bits(a.x, b.x);
        r.y = add_f32_bits(a.y, b.y);
        r.z = add_f32_bits(a.z, b.z);
        r.w = add_f32_bits(a.w, b.w);
    } else if (DT == 1) {
        r.x = add_bf16x2_bits(a.x, b.x);
        r.y = add_bf16x2_bits(a.y, b.y);
        r.z = add_bf16x2_bits(a.z, b.z);
        r.w = add_bf16x2_bits(a.w, b.w);
    } else {
        r.x = a.x + b.x;
        r.y = a.y + b.y;
        r.z = a.z + b.z;
        r.w = a.w + b.w;
    }
    return r;
}

} // namespace rc
