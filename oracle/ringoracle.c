/*
 * ringoracle.c -- the ORACLE for the ring collectives.  TEST INFRASTRUCTURE.
 *
 * A plain, slow, obviously correct CPU statement of what the ring collectives
 * compute.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may load this file's library; the product (the CUDA library and
 * its Python binding) never calls it and shares no code, header or helper with
 * it.
 *
 * Sources, cited by page title and section:
 *   [PALLAS]  "Pallas TPU Distributed Collectives 复习文档" (wqh011128 blog):
 *             s0.1 ring device model, s1 ppermute, s2 all_gather, s3 psum.
 *   [TPUBOOK] "TPU 与分布式通信原语" (fangpin gpu-hpc-book ch.09):
 *             section "reduce-scatter 与 all-gather", section "collective matmul".
 *   [PYPTO]   "全归约 3：Ring——每步大小恒定" (PyPTO distributed, step 10):
 *             sections "思路", "走读", "成本卡", "边界情况".
 *
 * Layout convention (shared by every routine, stated by the ring model of
 * [PALLAS] s0.1 and the symmetric-memory model of the Triton-distributed
 * semantics page): the P logical ranks are P slots; slot r starts at
 * base + r*stride bytes.  A chunk is N/P consecutive elements of a slot;
 * chunk k covers elements [k*c, (k+1)*c).
 *
 * Element types: ORC_F32 (IEEE binary32), ORC_BF16 (bfloat16 stored as the
 * upper 16 bits of a binary32), ORC_I32 (two's complement, wrapping),
 * ORC_TRACE (a fixed-width text cell that records the association tree of
 * every addition as "(left+own)"; used only to pin the schedule's order).
 *
 * Floating point: this file must be compiled without -ffast-math; the add of
 * two floats is then the IEEE round-to-nearest-even add, subnormals kept.
 *
 * Return value of every entry point: 0 on success, -1 on invalid arguments.
 *
 * Parity pins (what the tests check this file against) are listed per routine.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <stdio.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_I32 = 2, ORC_TRACE = 3 };

#define ORC_TRACE_W 192 /* bytes per ORC_TRACE cell, NUL-terminated text */

static size_t elem_size(int dtype)
{
    switch (dtype) {
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_I32: return 4;
    case ORC_TRACE: return ORC_TRACE_W;
    default: return 0;
    }
}

int orc_trace_width(void) { return ORC_TRACE_W; }

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> binary32, from the IEEE 754 round-to-nearest-even definition.
 * A bfloat16 is the upper half of a binary32.  Rounding keeps the upper 16
 * bits and adds one unit in the last kept place when the dropped 16 bits are
 * above half a unit, or exactly half a unit and the kept part is odd (ties to
 * even).  Adding 0x7FFF plus the kept part's lowest bit and truncating does
 * exactly that; a carry out of the significand correctly bumps the exponent
 * (and rounds the largest finite values up to infinity).  A NaN stays a NaN:
 * its upper half is kept and the quiet bit set, so truncation cannot turn it
 * into an infinity.
 * Pin: bit-equal to torch's CPU float32 -> bfloat16 conversion (RNE) on random
 * and special values.                                                        */
static uint16_t bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

int orc_bf16_from_f32(const float *in, uint16_t *out, size_t n)
{
    if ((!in || !out) && n) return -1;
    for (size_t i = 0; i < n; ++i) out[i] = bf16_rne(in[i]);
    return 0;
}

int orc_f32_from_bf16(const uint16_t *in, float *out, size_t n)
{
    if ((!in || !out) && n) return -1;
    for (size_t i = 0; i < n; ++i) out[i] = bf16_to_f32(in[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The reduction operator (+) of one hop, element by element:
 *   own <- partial_from_left (+) own
 * f32:   IEEE binary32 add.
 * bf16:  widen both to binary32, add in binary32, round the sum to bfloat16
 *        (each hop adds in fp32 and rounds the partial sum to bf16).
 * i32:   wrapping add, done in uint32_t so overflow is defined.
 * trace: own <- "(" partial "+" own ")".                                    */
static void hop_add(int dtype, void *own, const void *partial, size_t n)
{
    size_t i;
    switch (dtype) {
    case ORC_F32: {
        float *a = (float *)own;
        const float *b = (const float *)partial;
        for (i = 0; i < n; ++i) a[i] = b[i] + a[i];
        break;
    }
    case ORC_BF16: {
        uint16_t *a = (uint16_t *)own;
        const uint16_t *b = (const uint16_t *)partial;
        for (i = 0; i < n; ++i) a[i] = bf16_rne(bf16_to_f32(b[i]) + bf16_to_f32(a[i]));
        break;
    }
    case ORC_I32: {
        uint32_t *a = (uint32_t *)own;
        const uint32_t *b = (const uint32_t *)partial;
        for (i = 0; i < n; ++i) a[i] = b[i] + a[i];
        break;
    }
    case ORC_TRACE: {
        char *a = (char *)own;
        const char *b = (const char *)partial;
        char tmp[ORC_TRACE_W];
        for (i = 0; i < n; ++i) {
            int w = snprintf(tmp, sizeof tmp, "(%s+%s)", b + i * ORC_TRACE_W, a + i * ORC_TRACE_W);
            if (w < 0 || w >= ORC_TRACE_W) strcpy(tmp, "!overflow");
            memcpy(a + i * ORC_TRACE_W, tmp, ORC_TRACE_W);
        }
        break;
    }
    }
}

static char *slot_at(void *base, size_t stride, int r) { return (char *)base + (size_t)r * stride; }
static const char *cslot_at(const void *base, size_t stride, int r)
{
    return (const char *)base + (size_t)r * stride;
}

static int layout_ok(const void *base, size_t stride, int P, size_t n_elems, int dtype)
{
    size_t es = elem_size(dtype);
    if (es == 0 || P < 1) return 0;
    if (n_elems == 0) return 1;
    if (!base) return 0;
    if (P > 1 && stride < n_elems * es) return 0;
    return 1;
}

/* ------------------------------------------------------------------------ */
/* ppermute right shift ([PALLAS] s1, table in s1.4): every device sends its
 * shard to its right neighbour right = (r+1) % P, so device r ends with the
 * shard of its left neighbour:  dst_r = src_{(r-1+P) % P}.
 * Pin: the 4-device table D0:x3, D1:x0, D2:x1, D3:x2.                      */
int orc_ppermute_right(const void *src, size_t src_stride, void *dst, size_t dst_stride,
                       int P, size_t n, int dtype)
{
    if (!layout_ok(src, src_stride, P, n, dtype) || !layout_ok(dst, dst_stride, P, n, dtype)) return -1;
    size_t bytes = n * elem_size(dtype);
    for (int r = 0; r < P; ++r) {
        int left = (r - 1 + P) % P;
        memcpy(slot_at(dst, dst_stride, r), cslot_at(src, src_stride, left), bytes);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* all_gather, definition ([PALLAS] s2.1; [TPUBOOK] "reduce-scatter 与
 * all-gather"): every device ends with all shards in rank order,
 *   out_r[k] = in_k  for every k,  out slot r holding P*n elements.
 * Pin: the per-step slot table of [PALLAS] s2.5 via orc_all_gather_ring,
 * which must agree with this definition after its last step.               */
int orc_all_gather(const void *in, size_t in_stride, void *out, size_t out_stride,
                   int P, size_t n, int dtype)
{
    if (!layout_ok(in, in_stride, P, n, dtype) || !layout_ok(out, out_stride, P, (size_t)P * n, dtype))
        return -1;
    size_t bytes = n * elem_size(dtype);
    for (int r = 0; r < P; ++r)
        for (int k = 0; k < P; ++k)
            memcpy(slot_at(out, out_stride, r) + (size_t)k * bytes, cslot_at(in, in_stride, k), bytes);
    return 0;
}

/* all_gather as the ring schedule ([TPUBOOK] all_gather kernel; the same
 * order as [PALLAS] s2.4): each device first places its own shard at chunk
 * my_id of its output; then for step = 0 .. P-2 it receives from its left
 * neighbour the chunk recv_idx = (my_id - step - 1 + P) % P, which the left
 * neighbour sends as its send_idx = (left - step + P) % P.  Only the first
 * nsteps steps run (nsteps < 0: all), so the state after each step can be
 * compared with the slot table of [PALLAS] s2.5.  Chunks not yet received
 * are left as they were in `out`.
 * Messages are taken from every device's state before the step, then
 * applied, which is the lock-step reading of "receive from the left".      */
int orc_all_gather_ring(const void *in, size_t in_stride, void *out, size_t out_stride,
                        int P, size_t n, int dtype, int nsteps)
{
    if (!layout_ok(in, in_stride, P, n, dtype) || !layout_ok(out, out_stride, P, (size_t)P * n, dtype))
        return -1;
    size_t bytes = n * elem_size(dtype);
    if (bytes == 0) return 0;
    if (nsteps < 0 || nsteps > P - 1) nsteps = P - 1;
    for (int r = 0; r < P; ++r)
        memcpy(slot_at(out, out_stride, r) + (size_t)r * bytes, cslot_at(in, in_stride, r), bytes);
    char *msg = (char *)malloc((size_t)P * bytes);
    if (!msg) return -1;
    for (int step = 0; step < nsteps; ++step) {
        for (int r = 0; r < P; ++r) {
            int left = (r - 1 + P) % P;
            int send_idx = (left - step + P) % P;
            memcpy(msg + (size_t)r * bytes, slot_at(out, out_stride, left) + (size_t)send_idx * bytes, bytes);
        }
        for (int r = 0; r < P; ++r) {
            int recv_idx = (r - step - 1 + P) % P;
            memcpy(slot_at(out, out_stride, r) + (size_t)recv_idx * bytes, msg + (size_t)r * bytes, bytes);
        }
    }
    free(msg);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The ring all-reduce schedule of [PYPTO] "走读", on P slots of N elements,
 * chunk = N/P, in place.  Global step g runs 0 .. 2(P-1)-1; steps run past
 * nsteps are skipped (nsteps < 0: all), so partial states can be pinned.
 *
 * Reduce-scatter, P-1 rounds, s = 0 .. P-2 (signal row s):
 *     step          = s + 1
 *     left          = (my_rank - 1 + P) % P          (never negative)
 *     recv_add_idx  = (my_rank - step - 1 + P) % P
 *     left_send_idx = (left - step + P) % P
 *     local chunk recv_add_idx <- left's chunk left_send_idx (+) local chunk
 *   (the two indices are always equal: the chunk a device adds into is the
 *   one its left neighbour forwards).  After P-1 rounds device r holds the
 *   fully reduced chunk r.
 *
 * All-gather, P-1 rounds, t = 0 .. P-2 (signal rows P-1 .. 2(P-1)-1): the
 * page states it in words only: the reduced chunk keeps travelling round the
 * ring and every device copies the left neighbour's send chunk into its own
 * chunk.  Reading taken here (the plainest one, and the index rule of the
 * [TPUBOOK] all_gather): in round t the left neighbour sends the chunk it
 * completed or received last, send_idx = (left - t + P) % P, and the device
 * stores it at the same chunk index, so chunk (my_rank - 1 - t + P) % P.
 *
 * Messages of a round are collected from every device's state before the
 * round, then applied: a device always sees its left neighbour's state after
 * the previous round, as the signal handshake (wait on row s from the left,
 * notify row s+1 of the right after the store) enforces.
 *
 * The value this yields for chunk k, every element, on every device, is the
 * left fold that starts at device k+1 and ends with device k:
 *     R[k] = ((x_{k+1} (+) x_{k+2}) (+) ...) (+) x_k        (indices mod P)
 * (orc_ring_fold_at states that closed form; the tests pin the two together).
 *
 * Pins: integer-valued floats and i32 give the exact sum; the i32 bit-mask
 * test (x_r = 1<<r gives 2^P - 1 everywhere); the positional test; every
 * device bit-identical; P=2 is the plain two-term sum; the ORC_TRACE order
 * table for P=4 derived by hand from the index rules above.                */
int orc_ring_allreduce(void *bufs, size_t stride, int P, size_t N, int dtype, int nsteps)
{
    if (!layout_ok(bufs, stride, P, N, dtype)) return -1;
    if (N % (size_t)P) return -1;          /* [PYPTO]: SIZE must divide by the rank count */
    if (P == 1 || N == 0) return 0;         /* one rank: already reduced */
    size_t es = elem_size(dtype);
    size_t chunk = N / (size_t)P;
    size_t cbytes = chunk * es;
    int total = 2 * (P - 1);
    if (nsteps < 0 || nsteps > total) nsteps = total;
    char *msg = (char *)malloc((size_t)P * cbytes);
    if (!msg) return -1;
    int g = 0;
    /* reduce-scatter */
    for (int s = 0; s < P - 1 && g < nsteps; ++s, ++g) {
        int step = s + 1;
        for (int my_rank = 0; my_rank < P; ++my_rank) {
            int left = (my_rank - 1 + P) % P;
            int left_send_idx = (left - step + P) % P;
            memcpy(msg + (size_t)my_rank * cbytes,
                   slot_at(bufs, stride, left) + (size_t)left_send_idx * cbytes, cbytes);
        }
        for (int my_rank = 0; my_rank < P; ++my_rank) {
            int recv_add_idx = (my_rank - step - 1 + P) % P;
            hop_add(dtype, slot_at(bufs, stride, my_rank) + (size_t)recv_add_idx * cbytes,
                    msg + (size_t)my_rank * cbytes, chunk);
        }
    }
    /* all-gather */
    for (int t = 0; t < P - 1 && g < nsteps; ++t, ++g) {
        for (int my_rank = 0; my_rank < P; ++my_rank) {
            int left = (my_rank - 1 + P) % P;
            int send_idx = (left - t + P) % P;
            memcpy(msg + (size_t)my_rank * cbytes,
                   slot_at(bufs, stride, left) + (size_t)send_idx * cbytes, cbytes);
        }
        for (int my_rank = 0; my_rank < P; ++my_rank) {
            int recv_idx = (my_rank - 1 - t + P) % P;
            memcpy(slot_at(bufs, stride, my_rank) + (size_t)recv_idx * cbytes,
                   msg + (size_t)my_rank * cbytes, cbytes);
        }
    }
    free(msg);
    return 0;
}

/* Standalone ring reduce-scatter ([TPUBOOK] reduce_scatter kernel; the
 * reduce-scatter half of [PYPTO]): the same P-1 rounds, except that the last
 * round (s = P-2, where recv_add_idx = my_rank) writes its sum to out_r
 * instead of back into the slot, as the [TPUBOOK] kernel writes its last
 * reduced chunk to out_ref.  So out_r = R[r] (chunk r fully reduced), and
 * `bufs` is left holding the partial sums of rounds 0 .. P-3 (chunk r of slot
 * r keeps its input value).  P = 1: the reduction of one contributor is the
 * contributor, out_0 = chunk 0 of slot 0 (the pages are silent; plainest
 * reading).
 * Pins: out_r equals chunk r of orc_ring_allreduce's result bit for bit;
 * semantics D_b = sum over devices of block b ([PALLAS] s4.1); brute force.  */
int orc_reduce_scatter(void *bufs, size_t stride, void *out, size_t out_stride,
                       int P, size_t N, int dtype)
{
    if (!layout_ok(bufs, stride, P, N, dtype)) return -1;
    if (N % (size_t)P) return -1;
    size_t es = elem_size(dtype);
    size_t chunk = N / (size_t)P;
    if (!layout_ok(out, out_stride, P, chunk, dtype)) return -1;
    size_t cbytes = chunk * es;
    if (cbytes == 0) return 0;
    if (P == 1) {
        memcpy(out, bufs, cbytes);
        return 0;
    }
    char *msg = (char *)malloc((size_t)P * cbytes);
    if (!msg) return -1;
    for (int s = 0; s < P - 1; ++s) {
        int step = s + 1;
        for (int my_rank = 0; my_rank < P; ++my_rank) {
            int left = (my_rank - 1 + P) % P;
            int left_send_idx = (left - step + P) % P;
            memcpy(msg + (size_t)my_rank * cbytes,
                   slot_at(bufs, stride, left) + (size_t)left_send_idx * cbytes, cbytes);
        }
        for (int my_rank = 0; my_rank < P; ++my_rank) {
            int recv_add_idx = (my_rank - step - 1 + P) % P;
            char *own = slot_at(bufs, stride, my_rank) + (size_t)recv_add_idx * cbytes;
            if (s == P - 2) {
                char *dst = slot_at(out, out_stride, my_rank);
                memcpy(dst, own, cbytes);
                hop_add(dtype, dst, msg + (size_t)my_rank * cbytes, chunk);
            } else {
                hop_add(dtype, own, msg + (size_t)my_rank * cbytes, chunk);
            }
        }
    }
    free(msg);
    return 0;
}

/* Closed form of the ring fold at chosen element indices (see the comment of
 * orc_ring_allreduce): for element i of a slot, k = i / chunk, and
 *     R[k][i] = ((x_{k+1}[i] (+) x_{k+2}[i]) (+) ... (+) x_{k+P-1}[i]) (+) x_k[i]
 * computed one element at a time from the inputs x (never modified).  For
 * the commutative hop operator, x_{k+1} (+) x_{k+2} is the first hop's
 * x_{k+2} (+) x_{k+1}.  Lets the tests check sampled outputs of inputs too
 * large for the full simulation.  out holds nidx elements of dtype.
 * Pin: equal, bit for bit, to orc_ring_allreduce on random inputs.          */
int orc_ring_fold_at(const void *x, size_t stride, int P, size_t N, int dtype,
                     const int64_t *idx, size_t nidx, void *out)
{
    if (!layout_ok(x, stride, P, N, dtype)) return -1;
    if (N % (size_t)P) return -1;
    if ((!idx || !out) && nidx) return -1;
    size_t es = elem_size(dtype);
    size_t chunk = N / (size_t)P;
    for (size_t q = 0; q < nidx; ++q) {
        if (idx[q] < 0 || (size_t)idx[q] >= N) return -1;
        size_t i = (size_t)idx[q];
        int k = (int)(i / chunk);
        char *acc = (char *)out + q * es;
        memcpy(acc, cslot_at(x, stride, (k + 1) % P) + i * es, es);
        for (int j = 2; j <= P; ++j) {
            int src = (k + j) % P; /* j = P gives x_k, the last term */
            char own[ORC_TRACE_W];
            memcpy(own, cslot_at(x, stride, src) + i * es, es);
            hop_add(dtype, own, acc, 1); /* own <- acc (+) own */
            memcpy(acc, own, es);
        }
    }
    return 0;
}

/* Naive left-to-right sum S[i] = ((x_0 + x_1) + ...) + x_{P-1}, the
 * single-order reference that ring results are compared with under a
 * tolerance ([PYPTO] "边界情况": ring sums equal on every rank but differ
 * from a plain sum by reduction order, so compare with a tolerance).
 * f32 and bf16 inputs sum in binary32 (bf16 widened, no rounding to bf16),
 * out is float; i32 sums wrap, out is int32; out holds N elements.
 * Pin: exact for integer-valued inputs; within (P-1) 2^-24 sum|x| of the
 * correctly rounded sum (math.fsum) on random inputs.                       */
int orc_naive_sum(const void *x, size_t stride, int P, size_t N, int dtype, void *out)
{
    if (dtype == ORC_TRACE || !layout_ok(x, stride, P, N, dtype)) return -1;
    if (!out && N) return -1;
    for (size_t i = 0; i < N; ++i) {
        if (dtype == ORC_I32) {
            uint32_t acc = 0;
            for (int r = 0; r < P; ++r) {
                uint32_t v;
                memcpy(&v, cslot_at(x, stride, r) + i * 4, 4);
                acc += v;
            }
            memcpy((char *)out + i * 4, &acc, 4);
        } else {
            float acc = 0.0f;
            for (int r = 0; r < P; ++r) {
                float v;
                if (dtype == ORC_F32) {
                    memcpy(&v, cslot_at(x, stride, r) + i * 4, 4);
                } else {
                    uint16_t h;
                    memcpy(&h, cslot_at(x, stride, r) + i * 2, 2);
                    v = bf16_to_f32(h);
                }
                acc = (r == 0) ? v : acc + v;
            }
            memcpy((char *)out + i * 4, &acc, 4);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* psum: unidirectional rotate-and-accumulate all-reduce ([PALLAS] s3, the
 * psum kernel and the state table of s3.5).  Every device keeps a
 * two-slot communication buffer H[2] and an accumulator o (zeroed):
 *   prologue: device r writes x_r into slot 0 of its right neighbour.
 *   step t = 0 .. P-1 (working = t % 2, receiving = 1 - working):
 *     recv = own H[working];  the right neighbour's H[receiving] <- own
 *     H[working] (forward);  o <- o (+) recv.
 * After P steps o = (((0 (+) x_{r-1}) (+) x_{r-2}) ...) (+) x_r: every
 * device sums all inputs, each in its own rotated order, so fp results may
 * differ between devices (the page's point of contrast with the ring).
 * Messages of a step are taken from every device's state before the step.
 * x and out are P slots of n elements; h0/h1 (may be NULL) receive the
 * final H[0] / H[1] of every device (slots of n), for the state-table pin.
 * nsteps < 0 runs all P steps; the prologue always runs.  Unwritten H slots
 * are zero.  Pin: the table of [PALLAS] s3.5 (all buffers, every step),
 * exact integer sums, the per-device order via ORC_TRACE.                  */
int orc_psum(const void *x, size_t x_stride, void *out, size_t out_stride, int P, size_t n, int dtype,
             int nsteps, void *h0, void *h1)
{
    if (!layout_ok(x, x_stride, P, n, dtype) || !layout_ok(out, out_stride, P, n, dtype)) return -1;
    size_t es = elem_size(dtype);
    size_t bytes = n * es;
    if (bytes == 0) return 0;
    if (nsteps < 0 || nsteps > P) nsteps = P;
    char *H = (char *)calloc((size_t)P * 2, bytes);      /* H[r][slot] */
    char *o = (char *)calloc((size_t)P, bytes);
    char *snap = (char *)malloc((size_t)P * 2 * bytes);
    if (!H || !o || !snap) { free(H); free(o); free(snap); return -1; }
    if (dtype == ORC_TRACE)
        for (size_t i = 0; i < (size_t)P * n; ++i) strcpy(o + i * ORC_TRACE_W, "0");
    /* (an all-zero bit pattern is +0 for f32 / bf16 and 0 for i32) */
    for (int r = 0; r < P; ++r) {
        int right = (r + 1) % P;
        memcpy(H + ((size_t)right * 2 + 0) * bytes, cslot_at(x, x_stride, r), bytes);
    }
    for (int t = 0; t < nsteps; ++t) {
        int working = t % 2, receiving = 1 - working;
        memcpy(snap, H, (size_t)P * 2 * bytes);
        for (int r = 0; r < P; ++r) {
            int right = (r + 1) % P;
            const char *recv = snap + ((size_t)r * 2 + working) * bytes;
            memcpy(H + ((size_t)right * 2 + receiving) * bytes, recv, bytes);
        }
        for (int r = 0; r < P; ++r) {
            const char *recv = snap + ((size_t)r * 2 + working) * bytes;
            /* o <- o (+) recv, written as own <- partial (+) own with the
             * accumulator as the partial: copy, then add the received block */
            char *acc = o + (size_t)r * bytes;
            char *tmp = (char *)malloc(bytes);
            if (!tmp) { free(H); free(o); free(snap); return -1; }
            memcpy(tmp, recv, bytes);
            hop_add(dtype, tmp, acc, n);   /* tmp <- acc (+) recv */
            memcpy(acc, tmp, bytes);
            free(tmp);
        }
    }
    for (int r = 0; r < P; ++r) {
        memcpy(slot_at(out, out_stride, r), o + (size_t)r * bytes, bytes);
        if (h0) memcpy((char *)h0 + (size_t)r * bytes, H + ((size_t)r * 2 + 0) * bytes, bytes);
        if (h1) memcpy((char *)h1 + (size_t)r * bytes, H + ((size_t)r * 2 + 1) * bytes, bytes);
    }
    free(H);
    free(o);
    free(snap);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Bidirectional reduce-scatter ([PALLAS] s4, the psum_scatter kernel and the
 * state tables of s4.6).  Every device holds P blocks x_me[b] (block b =
 * elements [b*c, (b+1)*c), c = N/P); a block is split into a top half
 * (elements [0, c/2)) that travels LEFT and a bottom half ([c/2, c)) that
 * travels RIGHT.  Device me keeps a two-slot buffer H[2] (each slot one
 * block: top + bottom), an accumulator and its output o (block me).
 * The grid is (step = 0..P-1) x (phase = LEFT, RIGHT); with working =
 * step % 2, receiving = 1 - working, left_block = (me+step+1) % P,
 * right_block = (me-step-1) % P, in this order per iteration:
 *   first iteration (0, LEFT): o = 0; init_left: the LEFT neighbour's
 *     H[working].top <- x_me[me].top, completed before the local update;
 *     init_right: the RIGHT neighbour's H[working].bottom <- x_me[me].bottom.
 *   other LEFT phases:  send_right: RIGHT neighbour's H[working].bottom <-
 *     own H[receiving].bottom.
 *   RIGHT phases:       send_left: LEFT neighbour's H[receiving].top <- own
 *     H[working].top.
 *   local update of the current half (top in LEFT, bottom in RIGHT):
 *     accum <- H[working].half; unless last step: accum <- accum (+)
 *     x_me[left_block or right_block].half; H[working].half <- accum; on the
 *     last step o.half <- accum.
 * Transfers started in an iteration land at its end (the page waits on them
 * before the next iteration); they never touch the half being updated.
 * Result: o_me.top = ((x_me + x_{me-1}) + ...) + x_{me+1} over block me's
 * top halves, o_me.bottom = ((x_me + x_{me+1}) + ...) + x_{me-1} over its
 * bottom halves.
 * out: P slots of c elements.  iters (< 0: all 2P) limits the iterations run;
 * state (may be NULL) receives, per device, H0.top H0.bot H1.top H1.bot
 * accum o.top o.bot as [P][7][hmax] elements, hmax = c - c/2 (top halves
 * padded); for ORC_TRACE, never-written cells stay empty.
 * Pin: the eight state tables of [PALLAS] s4.6; block sums in integers.    */
int orc_reduce_scatter_bidir(const void *x, size_t x_stride, void *out, size_t out_stride, int P, size_t N,
                             int dtype, int iters, void *state)
{
    if (!layout_ok(x, x_stride, P, N, dtype)) return -1;
    if (N % (size_t)P) return -1;
    size_t es = elem_size(dtype), c = N / (size_t)P;
    if (!layout_ok(out, out_stride, P, c, dtype)) return -1;
    if (c == 0) return 0;
    size_t half = c / 2, hmax = c - half;     /* top: [0, half), bottom: [half, c) */
    size_t cb = c * es;
    char *H = (char *)calloc((size_t)P * 2, cb);    /* H[me][slot] block */
    char *acc = (char *)calloc((size_t)P, hmax * es);
    char *o = (char *)calloc((size_t)P, cb);
    char *tmp = (char *)malloc(hmax * es);
    if (!H || !acc || !o || !tmp) { free(H); free(acc); free(o); free(tmp); return -1; }
#define HB(me, slot) (H + ((size_t)(me) * 2 + (slot)) * cb)
#define XB(me, b) (cslot_at(x, x_stride, (me)) + (size_t)(b) * cb)
    int total = 2 * P;
    if (iters < 0 || iters > total) iters = total;
    for (int it = 0; it < iters; ++it) {
        int step = it / 2, phase = it % 2;           /* phase 0 = LEFT, 1 = RIGHT */
        int working = step % 2, receiving = 1 - working;
        int is_first = (step == 0 && phase == 0), is_last = (step == P - 1);
        if (is_first)                                /* init_left, completed before the local update */
            for (int me = 0; me < P; ++me)
                memcpy(HB((me - 1 + P) % P, working), XB(me, me), half * es);
        /* transfers started now, landing at the end of the iteration (taken from the current state) */
        char *pending = (char *)malloc((size_t)P * cb);
        if (!pending) { free(H); free(acc); free(o); free(tmp); return -1; }
        for (int me = 0; me < P; ++me) {
            char *msg = pending + (size_t)me * cb;
            if (is_first)
                memcpy(msg, XB(me, me) + half * es, hmax * es);             /* bottom of x_me[me] */
            else if (phase == 0)
                memcpy(msg, HB(me, receiving) + half * es, hmax * es);      /* own H[receiving].bottom */
            else
                memcpy(msg, HB(me, working), half * es);                     /* own H[working].top */
        }
        /* local update of the current half */
        for (int me = 0; me < P; ++me) {
            size_t off = phase == 0 ? 0 : half, len = phase == 0 ? half : hmax;
            int blk = phase == 0 ? (me + step + 1) % P : ((me - step - 1) % P + P) % P;
            char *a = acc + (size_t)me * hmax * es;
            memcpy(a, HB(me, working) + off * es, len * es);
            if (!is_last) {
                memcpy(tmp, XB(me, blk) + off * es, len * es);
                hop_add(dtype, tmp, a, len);      /* tmp <- accum (+) x */
                memcpy(a, tmp, len * es);
            }
            memcpy(HB(me, working) + off * es, a, len * es);
            if (is_last) memcpy(o + (size_t)me * cb + off * es, a, len * es);
        }
        /* land the transfers */
        for (int me = 0; me < P; ++me) {
            const char *msg = pending + (size_t)me * cb;
            if (is_first || phase == 0)
                memcpy(HB((me + 1) % P, working) + half * es, msg, hmax * es);
            else
                memcpy(HB((me - 1 + P) % P, receiving), msg, half * es);
        }
        free(pending);
    }
    for (int me = 0; me < P; ++me) {
        memcpy(slot_at(out, out_stride, me), o + (size_t)me * cb, cb);
        if (state) {
            char *st = (char *)state + (size_t)me * 7 * hmax * es;
            memcpy(st + 0 * hmax * es, HB(me, 0), half * es);
            memcpy(st + 1 * hmax * es, HB(me, 0) + half * es, hmax * es);
            memcpy(st + 2 * hmax * es, HB(me, 1), half * es);
            memcpy(st + 3 * hmax * es, HB(me, 1) + half * es, hmax * es);
            memcpy(st + 4 * hmax * es, acc + (size_t)me * hmax * es, hmax * es);
            memcpy(st + 5 * hmax * es, o + (size_t)me * cb, half * es);
            memcpy(st + 6 * hmax * es, o + (size_t)me * cb + half * es, hmax * es);
        }
    }
#undef HB
#undef XB
    free(H);
    free(acc);
    free(o);
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* All-gather + matmul ([TPUBOOK] "collective matmul": gather the row shards,
 * then multiply by the local weight, bf16 result as its _matmul_bf16 casts).
 *
 * orc_ag_gather: A_g rows [r*M_r, (r+1)*M_r) = shard r (rank order, the
 * all_gather definition applied to row blocks).  Shards are bf16 [M_r][K]
 * row-major, slot r at a_shards + r*stride bytes; A_g is [P*M_r][K].       */
int orc_ag_gather(const void *a_shards, size_t stride, int P, int M_r, int K, void *a_gathered)
{
    if (P < 1 || M_r < 0 || K < 0) return -1;
    size_t shard_bytes = (size_t)M_r * (size_t)K * 2;
    if (shard_bytes == 0) return 0;
    if (!a_shards || !a_gathered || (P > 1 && stride < shard_bytes)) return -1;
    for (int r = 0; r < P; ++r)
        memcpy((char *)a_gathered + (size_t)r * shard_bytes, cslot_at(a_shards, stride, r), shard_bytes);
    return 0;
}

/* C = A_g . B^T at the rows x cols grid given (rows/cols NULL: all), with
 * A_g bf16 [M][K] row-major and B bf16 [N][K] row-major (the weight stored
 * one output feature per row), so C[m][n] = sum_k A_g[m][k] * B[n][k].
 * Each product and the sum are formed in binary64 (bf16 products are exact
 * in binary64; the sum is far more accurate than any binary32 order), then
 * out_f64 gets the binary64 sum and out_bf16 its bf16 rounding (through
 * binary32: the binary64 sum is first rounded to binary32 by the C
 * conversion, then to bf16; see the tolerance derivation for why this double
 * rounding stays within the bound).  Outputs are [nrows][ncols]; either may
 * be NULL.  abs_out (may be NULL) gets sum_k |A_g[m][k] * B[n][k]| for the
 * error bound.
 * Pins: numpy float64 matmul of the same bf16 values; a tiny hand example.  */
int orc_gemm_bf16_at(const uint16_t *A, const uint16_t *B, int M, int N, int K,
                     const int64_t *rows, size_t nrows, const int64_t *cols, size_t ncols,
                     double *out_f64, uint16_t *out_bf16, double *abs_out)
{
    if (M < 0 || N < 0 || K < 0 || !A || !B) return -1;
    size_t nr = rows ? nrows : (size_t)M;
    size_t nc = cols ? ncols : (size_t)N;
    for (size_t a = 0; a < nr; ++a) {
        int64_t m = rows ? rows[a] : (int64_t)a;
        if (m < 0 || m >= M) return -1;
        for (size_t b = 0; b < nc; ++b) {
            int64_t n = cols ? cols[b] : (int64_t)b;
            if (n < 0 || n >= N) return -1;
            double acc = 0.0, aacc = 0.0;
            const uint16_t *arow = A + (size_t)m * (size_t)K;
            const uint16_t *brow = B + (size_t)n * (size_t)K;
            for (int k = 0; k < K; ++k) {
                double p = (double)bf16_to_f32(arow[k]) * (double)bf16_to_f32(brow[k]);
                acc += p;
                aacc += p < 0 ? -p : p;
            }
            if (out_f64) out_f64[a * nc + b] = acc;
            if (out_bf16) out_bf16[a * nc + b] = bf16_rne((float)acc);
            if (abs_out) abs_out[a * nc + b] = aacc;
        }
    }
    return 0;
}
