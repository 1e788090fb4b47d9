/*
 * ringcoll.h -- C ABI of libringcoll.so: ring collectives over P logical
 * ranks that live in one GPU's HBM.
 *
 * Model.  The P ranks are P symmetric slots of device memory: slot r starts
 * at base + r*stride bytes, so the symmetric-memory lookup symm_at(ptr, r) of
 * "Triton-distributed 语义" (section "对称内存模型") is pointer arithmetic.
 * Ranks form the ring of "Pallas TPU Distributed Collectives 复习文档",
 * section 0.1: right = (r+1) % P, left = (r-1+P) % P.  A chunk is N/P
 * consecutive elements of a slot; chunk k covers elements [k*N/P, (k+1)*N/P).
 *
 * Conventions shared by every entry point:
 *   - Pointers named *_base and the buffers of ag_gemm are DEVICE pointers
 *     owned by the caller; the library never frees or keeps them.
 *   - *_stride arguments are in BYTES; a stride must be at least the bytes
 *     a slot uses (checked) and slots must not overlap each other.
 *   - dtype is an rc_dtype value; element sizes: f32 4, bf16 2, i32 4 bytes.
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call is asynchronous on it: the return value reports
 *     argument validation and launch errors only; errors raised on the device
 *     (a bounded wait that ran out) are read with ring_status().
 *   - Alignment: slot bases and strides must be multiples of the element
 *     size (RC_ERR_INVALID otherwise).  Kernels move the body of every range
 *     in 32-byte vectors when source and destination share their offset
 *     modulo 32 bytes (always, for 32-byte multiple strides), with element-wise
 *     heads and tails; other layouts run element-wise.
 *   - Degenerate sizes: n = 0 or N = 0 does nothing and returns RC_OK.
 *   - The library owns one signal workspace per device, created on the first
 *     call on that device (a cudaMalloc and a synchronous zeroing), grown on
 *     demand and released by ring_finalize().  Make the first call (at the
 *     largest P used) before capturing calls into a CUDA graph.  Calls that
 *     share a device's workspace must not run concurrently: issue them on one
 *     stream, or order the streams.  Every collective that signals also has
 *     an _ex variant taking a caller-owned workspace instead (sized by its
 *     *_workspace_bytes function, zeroed once before first use); calls with
 *     different workspaces may run concurrently on different streams, and a
 *     device timeout of such a call is read with ring_status_ex().
 *   - Return values are rc_status codes; ring_last_error() describes the most
 *     recent failure of the calling thread.
 *   - NaN.  The floating-point collectives are bit-identical to the fold
 *     orders stated below for every element whose result is not a NaN.  An
 *     element whose result is a NaN (a NaN input is folded into it, or +inf
 *     and -inf meet in one hop add) is a NaN here as well, but its sign and
 *     payload are unspecified: the hardware add returns its own NaN pattern,
 *     not one of the operands'.  Integer data has no such exception.
 */
#ifndef RINGCOLL_H
#define RINGCOLL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RC_F32 = 0, RC_BF16 = 1, RC_I32 = 2 } rc_dtype;

typedef enum {
    RC_OK = 0,
    RC_ERR_INVALID = 1,     /* bad argument, detected on the host before any launch */
    RC_ERR_CUDA = 2,        /* a CUDA runtime call failed (message in ring_last_error) */
    RC_ERR_TIMEOUT = 3,     /* a device-side bounded wait ran out (from ring_status) */
    RC_ERR_UNSUPPORTED = 4, /* no CUDA device, wrong architecture, or grid cannot be co-resident */
    RC_ERR_NOMEM = 5        /* the signal workspace could not be allocated */
} rc_status;

#define RC_MAX_P 64 /* largest number of logical ranks */

/* Layout of the weight B of ag_gemm: [N][K] (one output feature per row, the
 * nn.Linear layout) or [K][N] (the x @ W layout of "TPU 与分布式通信原语",
 * section "collective matmul"). */
typedef enum { RC_B_NK = 0, RC_B_KN = 1 } rc_b_layout;

/*
 * ring_ppermute_right -- right shift by one rank.
 * "Pallas TPU Distributed Collectives 复习文档", section 1 (lax.ppermute):
 * every rank sends its shard to its right neighbour, so rank r ends with
 * the shard of its left neighbour:  dst_r[i] = src_{(r-1+P)%P}[i], i < n.
 * src slots: [n] elements at src_base + r*src_stride (read only).
 * dst slots: [n] elements at dst_base + r*dst_stride (written).
 * The src and dst regions must not overlap (RC_ERR_INVALID otherwise).
 * P = 1 copies slot 0 to slot 0 of dst.
 */
int ring_ppermute_right(const void *src_base, size_t src_stride, void *dst_base, size_t dst_stride,
                        int P, size_t n, int dtype, void *stream);

/*
 * ring_all_gather -- every rank ends with every rank's shard, in rank order.
 * "Pallas TPU Distributed Collectives 复习文档", section 2 (lax.all_gather),
 * and "TPU 与分布式通信原语", section "reduce-scatter 与 all-gather": each rank
 * first places its own shard, then in ring step t = 0..P-2 copies from its
 * left neighbour the chunk (r-t-1+P)%P.
 * Result: out_r[k*n + i] = in_k[i] for every k < P, i < n.
 * in slots:  [n] elements at in_base + r*in_stride (read only).
 * out slots: [P*n] elements at out_base + r*out_stride (written).
 * in and out must not overlap.
 */
int ring_all_gather(const void *in_base, size_t in_stride, void *out_base, size_t out_stride,
                    int P, size_t n, int dtype, void *stream);

/*
 * ring_all_gather_ex -- ring_all_gather with a caller-owned signal workspace:
 * DEVICE memory of ws_bytes bytes, 16-byte aligned, zeroed once before its
 * first use and otherwise left to the library; calls sharing one must be
 * stream-ordered, calls with different workspaces may run concurrently
 * (re-zero it, with no call in flight, before about 2^30 calls).  ws_bytes
 * below ring_all_gather_workspace_bytes(P, n, dtype) gives RC_ERR_INVALID;
 * device timeouts are read with ring_status_ex(workspace, stream).
 * Arguments, validation and result as ring_all_gather.
 */
int ring_all_gather_ex(const void *in_base, size_t in_stride, void *out_base, size_t out_stride, int P, size_t n,
                       int dtype, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes ring_all_gather_ex needs for (P, n, dtype) on the current
 * device; 0 for invalid arguments or when no sm_103 device is current. */
size_t ring_all_gather_workspace_bytes(int P, size_t n, int dtype);

/*
 * ring_reduce_scatter -- rank r ends with the sum over ranks of chunk r.
 * "TPU 与分布式通信原语", section "reduce-scatter 与 all-gather" (the ring
 * reduce-scatter kernel, whose last step writes out_ref), with the round
 * indices of "全归约 3：Ring——每步大小恒定", section "走读": in round
 * s = 0..P-2 rank r adds its left neighbour's chunk (r-s-2+P)%P into its own
 * chunk of that index; the last round writes the sum to out_r instead.
 * Result: out_r = R[r], where for chunk k
 *     R[k] = ((x_{k+1} + x_{k+2}) + ... + x_{k+P-1}) + x_k   (indices mod P)
 * with "+" the element type's hop add (f32: IEEE binary32 add; bf16: add in
 * binary32, round the partial sum to bf16 at every hop; i32: wrapping add).
 * NaN results: bit-identity excludes them, see "NaN" above.
 * bufs slots: [N] elements at bufs_base + r*bufs_stride; CLOBBERED: their
 *     contents are undefined after the call (they hold partial sums, and the
 *     L2 lines of partials that are dead are dropped without write-back).
 * out slots:  [N/P] elements at out_base + r*out_stride (written); out must
 *     not overlap bufs.
 * N must be a multiple of P ("SIZE 必须能被 rank 数量整除", same page);
 * RC_ERR_INVALID otherwise.  P = 1 copies chunk 0 to out.
 */
int ring_reduce_scatter(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride,
                        int P, size_t N, int dtype, void *stream);

/*
 * ring_reduce_scatter_ex -- ring_reduce_scatter with a caller-owned signal
 * workspace (rules as for ring_all_gather_ex; size from
 * ring_reduce_scatter_workspace_bytes).  Arguments, validation and result as
 * ring_reduce_scatter.
 */
int ring_reduce_scatter_ex(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P, size_t N,
                           int dtype, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes ring_reduce_scatter_ex needs for (P, N, dtype) on the
 * current device; 0 for invalid arguments or no sm_103 device. */
size_t ring_reduce_scatter_workspace_bytes(int P, size_t N, int dtype);

/*
 * ring_reduce_scatter_bidir -- bidirectional reduce-scatter of "Pallas TPU
 * Distributed Collectives 复习文档", section 4 (psum_scatter): every chunk k
 * (a block of c = N/P elements) is split into a top half, elements
 * [0, c/2), whose partial sums travel LEFT round the ring, and a bottom half,
 * [c/2, c), whose partial sums travel RIGHT; both start at rank k with its
 * own contribution and are delivered to rank k after P-1 additions.
 * Result: out_r = block r summed over ranks, with
 *     top:    ((x_r + x_{r-1}) + x_{r-2}) + ... + x_{r+1}
 *     bottom: ((x_r + x_{r+1}) + x_{r+2}) + ... + x_{r-1}   (indices mod P)
 * ("+" the element type's hop add), the order of the page's state tables.
 * NaN results: bit-identity excludes them, see "NaN" above.
 * In round s = 0..P-2 every rank adds its own contribution to the partial
 * its upstream neighbour holds; round P-2 completes each half at the rank
 * one hop before its owner, which stores it straight into the owner's out
 * slot (the page's last hop, a plain transfer, is folded into that store).
 * bufs slots: [N] elements at bufs_base + r*bufs_stride; CLOBBERED (contents
 *     undefined afterwards, as for ring_reduce_scatter).
 * out slots:  [N/P] elements at out_base + r*out_stride (written).
 * N must be a multiple of P (RC_ERR_INVALID otherwise).  P = 1 copies.
 */
int ring_reduce_scatter_bidir(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P,
                              size_t N, int dtype, void *stream);

/*
 * ring_reduce_scatter_bidir_ex -- ring_reduce_scatter_bidir with a
 * caller-owned signal workspace (rules as for ring_all_gather_ex; size from
 * ring_reduce_scatter_bidir_workspace_bytes).
 */
int ring_reduce_scatter_bidir_ex(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P,
                                 size_t N, int dtype, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes ring_reduce_scatter_bidir_ex needs; 0 for invalid
 * arguments or no sm_103 device. */
size_t ring_reduce_scatter_bidir_workspace_bytes(int P, size_t N, int dtype);

/*
 * ring_allreduce -- in-place ring all-reduce: reduce-scatter (P-1 rounds)
 * then all-gather (P-1 rounds), 2(P-1) steps of one chunk each.
 * "全归约 3：Ring——每步大小恒定", sections "思路" and "走读":
 *   left = (r-1+P)%P; round s of reduce-scatter (signal row s) waits for the
 *   left neighbour, adds its chunk left_send_idx = (left-s-1+P)%P into the
 *   local chunk recv_add_idx = (r-s-2+P)%P (the same index), then signals
 *   the right neighbour on row s+1; all-gather round t (rows P-1..2P-3)
 *   copies the left neighbour's chunk (r-1-t+P)%P into the local chunk.
 * Synchronisation is neighbour-local (per-step signal rows, release/acquire),
 * with no grid-wide barrier.
 * Result: every slot holds R[0] | R[1] | ... | R[P-1] (R as for
 * ring_reduce_scatter), bit-identical on every rank (NaN results: see "NaN"
 * above; they are NaN on every rank).
 * bufs slots: [N] elements at bufs_base + r*stride, read and written in place.
 * N must be a multiple of P (RC_ERR_INVALID otherwise).  P = 1 is a no-op.
 */
int ring_allreduce(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *stream);

/*
 * ring_allreduce_ex -- ring_allreduce with a caller-owned signal workspace,
 * so that calls on different streams can run concurrently (each with its own
 * workspace) and no library allocation happens.  Arguments, validation and
 * result as ring_allreduce, plus:
 *   workspace: DEVICE memory of ws_bytes bytes, 16-byte aligned, owned by the
 *     caller, zeroed (e.g. cudaMemset 0) once before its first use and not
 *     modified otherwise.  Calls sharing a workspace must be stream-ordered;
 *     each call advances the epoch kept in it, so re-zero it (while no call is
 *     in flight) before about 2^30 calls.
 *   ws_bytes: at least ring_allreduce_workspace_bytes(P, N, dtype) for the
 *     current device (RC_ERR_INVALID otherwise).
 * Device-side timeouts are recorded in the workspace: read (and clear) them
 * with ring_status_ex(workspace, stream); ring_status() does not see them.
 * (The pages' signals live in per-rank signal buffers; this variant lets the
 * caller place them.)
 */
int ring_allreduce_ex(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *workspace, size_t ws_bytes,
                      void *stream);

/* Bytes of workspace ring_allreduce_ex needs for (P, N, dtype) on the current
 * device; 0 for invalid arguments or when no sm_103 device is current. */
size_t ring_allreduce_workspace_bytes(int P, size_t N, int dtype);

/*
 * ring_allreduce_fused -- the ring all-reduce's result in a single pass.
 * Same arguments, validation and result as ring_allreduce, bit for bit:
 * every element of chunk k becomes R[k] = ((x_{k+1} + x_{k+2}) + ...) + x_k,
 * the fold order that the reduce-scatter rounds of "全归约 3：Ring——每步大小恒定"
 * (section "走读") produce.  Instead of 2(P-1) ring steps over HBM, each
 * element position of all P slots is read once, folded on chip and written
 * to all P slots: 2*P*N*e bytes, the minimum for an all-reduce.  Uses no
 * signal workspace.  NaN results: as for ring_allreduce.
 */
int ring_allreduce_fused(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *stream);

/*
 * ring_psum -- rotate-and-accumulate all-reduce of "Pallas TPU Distributed
 * Collectives 复习文档", section 3 (psum): every rank starts an accumulator at
 * zero and, in each of P steps, adds the block that arrives from its left
 * neighbour, so rank r ends with
 *     o_r = (((0 + x_{r-1}) + x_{r-2}) + ...) + x_r       (indices mod P)
 * ("+" the element type's hop add).  Each rank folds in its own order, so
 * floating-point results may differ between ranks (unlike ring_allreduce).
 * NaN results: bit-identity excludes them, see "NaN" above.
 * bufs slots: [n] elements at bufs_base + r*stride, replaced by o_r in place.
 * n need not be a multiple of P.  P = 1: o_0 = 0 + x_0.
 */
int ring_psum(void *bufs_base, size_t stride, int P, size_t n, int dtype, void *stream);

/*
 * ring_allreduce_host -- ring_allreduce on inputs held in HOST memory:
 * copies slot r of h_in (host, [N] elements at h_in + r*h_in_stride) into
 * device slot r of d_bufs, runs the all-reduce there, and copies the result
 * of every slot back to h_out (host, may equal h_in).  d_bufs is caller-owned
 * device scratch of P slots (d_stride bytes apart).  Host buffers should be
 * page-locked (cudaHostAlloc / pinned) for the copies to be asynchronous.
 * From 128 MiB of slots on, the work runs in segments of about 64 MiB -- segment q is the
 * same sub-range of every chunk, so each element keeps its chunk and its
 * fold order and the result is the same bit for bit -- with the
 * host-to-device copies on one library-owned stream, the ring launches on
 * `stream` and the device-to-host copies on a second library-owned stream,
 * ordered by events, so both copy directions and the kernels overlap.  All
 * of it is ordered after earlier work on `stream`, and `stream` waits for
 * all of it: h_out is valid once `stream` completes.  Same validation and
 * result as ring_allreduce (device slot base and stride must be multiples of
 * the element size).
 */
int ring_allreduce_host(const void *h_in, size_t h_in_stride, void *h_out, size_t h_out_stride,
                        void *d_bufs, size_t d_stride, int P, size_t N, int dtype, void *stream);

/*
 * ag_gemm -- all-gather of row shards fused with a matmul, seen from rank
 * `rank`.  "TPU 与分布式通信原语", section "collective matmul" (all-gather then
 * local matmul, bf16 result), with the producer/consumer tiles, per-tile
 * wait and rank-swizzled tile order of "Triton-distributed 语义", sections
 * "生产者-消费者模型", "AllGather + GEMM 重叠", "线程块交织".
 * a_shards: bf16 [M_r][K] row-major per rank, slot r at a_shards + r*a_stride.
 * a_gathered: bf16 [P*M_r][K] row-major (written): rows [r*M_r, (r+1)*M_r)
 *     are shard r (the all-gather result, bit-exact copy).
 * B: bf16 [N][K] row-major (one output feature per row, the nn.Linear weight
 *     layout), read only.
 * C: bf16 [P*M_r][N] row-major (written): C = A_g . B^T, products summed in
 *     binary32, rounded once to bf16.
 * Requirements (RC_ERR_INVALID otherwise): 0 <= rank < P, M_r % 128 == 0,
 * N % 256 == 0, K % 64 == 0, all pointers 16-byte aligned, a_stride a
 * multiple of 16, no overlap between outputs and inputs.
 */
int ag_gemm(const void *a_shards, size_t a_stride, void *a_gathered, const void *B, void *C,
            int P, int rank, int M_r, int N, int K, void *stream);

/*
 * ag_gemm_kn -- ag_gemm with the weight stored [K][N] row-major (B[k][n] at
 * B + (k*N + n)*2 bytes), the layout of the page's x @ W1: C = A_g . B.  The
 * tensor cores read B as an MN-major operand straight from this layout (no
 * transpose pass).  Same requirements, result and rounding as ag_gemm; the
 * products are the same, so C is the same bit for bit as ag_gemm with the
 * transposed weight.
 */
int ag_gemm_kn(const void *a_shards, size_t a_stride, void *a_gathered, const void *B, void *C,
               int P, int rank, int M_r, int N, int K, void *stream);

/*
 * ag_gemm_ex -- ag_gemm with the weight layout as an argument (b_layout: an
 * rc_b_layout value; RC_ERR_INVALID otherwise) and a caller-owned workspace
 * holding the launch epoch, the status header and one ready flag per 16
 * gathered rows (rules as for ring_all_gather_ex; size from
 * ag_gemm_workspace_bytes(P, M_r)).  With different workspaces, ag_gemm_ex
 * calls may be issued on different streams; each launch fills the GPU, so
 * concurrent calls mostly run one after the other.  Arguments, validation and
 * result as ag_gemm (RC_B_NK) or ag_gemm_kn (RC_B_KN).
 */
int ag_gemm_ex(const void *a_shards, size_t a_stride, void *a_gathered, const void *B, int b_layout, void *C, int P,
               int rank, int M_r, int N, int K, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes ag_gemm_ex needs: 128 + 4 * P * M_r / 16; 0 when P or M_r
 * is invalid (M_r must be a multiple of 128). */
size_t ag_gemm_workspace_bytes(int P, int M_r);

/*
 * gemm_rs -- matmul followed by a ring reduce-scatter over output columns.
 * "TPU 与分布式通信原语", section "collective matmul" (matmul-reduce-scatter:
 * each rank's partial product is cast to bf16, laid out chunk-major by output
 * columns and reduce-scattered round the ring), overlapped as in
 * "Triton-distributed 语义", section "GEMM + ReduceScatter 重叠": here each
 * output tile's partial products are folded in the GEMM epilogue, so partial
 * products never reach memory.
 * A: bf16 [M][K] row-major per rank, slot r at A + r*a_stride (activations).
 * B: bf16 [N][K] row-major per rank, slot r at B + r*b_stride (row shard of
 *    the weight, one output feature per row).
 * out: bf16 [M][N/P] row-major per rank, slot r at out + r*out_stride
 *    (written): rank r's column chunk, columns [r*N/P, (r+1)*N/P), of
 *        R = ((C_{r+1} + C_{r+2}) + ...) + C_r,   C_q = bf16(A_q . B_q^T)
 *    with C_q accumulated in binary32 and rounded once, and "+" the bf16 hop
 *    add of ring_reduce_scatter -- the ring reduce-scatter of the chunk-major
 *    partial products.
 * Requirements (RC_ERR_INVALID otherwise): M % 128 == 0, K % 64 == 0, N a
 * multiple of 256*P, pointers and strides 16-byte aligned, out not
 * overlapping A or B.
 */
int gemm_rs(const void *A, size_t a_stride, const void *B, size_t b_stride, void *out, size_t out_stride,
            int P, int M, int N, int K, void *stream);

/*
 * gemm_rs_ex -- gemm_rs with a caller-owned workspace, which holds only the
 * launch's status header (rules as for ring_all_gather_ex; size from
 * gemm_rs_workspace_bytes).  Arguments, validation and result as gemm_rs.
 */
int gemm_rs_ex(const void *A, size_t a_stride, const void *B, size_t b_stride, void *out, size_t out_stride, int P,
               int M, int N, int K, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes gemm_rs_ex needs (the 128-byte header); 0 for invalid
 * arguments. */
size_t gemm_rs_workspace_bytes(int P, int M, int N, int K);

/*
 * ring_status -- waits for `stream`, then returns and clears the device
 * status of the library's own signal areas on the calling device: the
 * workspace of the regular entry points and the fixed array of
 * ring_allreduce_noalloc.  RC_OK, or RC_ERR_TIMEOUT when a bounded wait in a
 * kernel ran out (ring_last_error() then names the rank, step and slice that
 * gave up, and says whether it was an allocation-free call).  A timed-out
 * call leaves its outputs undefined; later calls are unaffected.  Reading the
 * status allocates nothing (a copy to host stack memory and a memset, both
 * on `stream`).
 */
int ring_status(void *stream);

/*
 * ring_status_ex -- ring_status for a caller-owned workspace (the one given
 * to an _ex entry point): waits for `stream`, then returns and clears the
 * status recorded in `workspace` (DEVICE pointer, 16-byte aligned; null or
 * misaligned gives RC_ERR_INVALID).  RC_OK or RC_ERR_TIMEOUT as above.
 */
int ring_status_ex(void *workspace, void *stream);

/* Message describing the calling thread's most recent error ("" if none). */
const char *ring_last_error(void);

/* Bound on every device-side wait, in milliseconds (1..600000; initial value
 * from the environment variable RC_TIMEOUT_MS, else 2000). */
int ring_set_timeout_ms(unsigned ms);

/*
 * Slices per rank for the ring kernels (0 = automatic; initial value from the
 * environment variable RC_SLICES, else 0).  Slice j of every chunk is an
 * independent ring with its own signals; the grid is P x slices co-resident
 * thread blocks.  Values above the co-residency limit are capped.
 *
 * Other environment settings, read once: RC_DEBUG_SERIAL=1 makes every step
 * of a ring launch also wait for all blocks of the launch (a bounded grid
 * barrier; for debugging synchronisation, results are unchanged);
 * RC_AG_BULK=0 / 1 moves the all-gather steps of every collective with
 * vector copies / bulk copies (default: vector in the all-reduce, bulk in the
 * all-gather); RC_L2_LIVE_BYTES sets the chunk-segment budget; RC_HOST_SEGMENT_BYTES
 * the host entry point's segment size; RC_GEMM_PAIRS=0 keeps the one-CTA
 * GEMM kernels; RC_RING_STAGGER=G (default 3, 1 = off) starts slice j of a
 * ring all-reduce or reduce-scatter (j % G) times a fifth of its first
 * step's estimated time later; RC_RING_PAIR=0 keeps the one-rank-per-block
 * ring kernel at even P as well; RC_PAIR_SMEM sets the bytes of a slice's
 * head that the two-rank kernel hands over in shared memory per block;
 * RC_FOLD_BLOCKS sets the blocks per SM of the single-pass all-reduces
 * (default max(1, 8/P)).
 */
int ring_set_slices(int slices);

/*
 * Test hook for failure detection: the next ring launch (ring_all_gather,
 * ring_reduce_scatter, ring_reduce_scatter_bidir, ring_allreduce,
 * ring_allreduce_ex or ring_allreduce_noalloc) on any thread skips the
 * notify that rank `rank` would send after global step `step`, in every
 * slice.  Its neighbour's bounded wait then runs out and ring_status() (or
 * ring_status_ex() for a caller's workspace) reports RC_ERR_TIMEOUT; no
 * fault is raised and the device stays usable.  Where two ranks share a
 * thread block (the all-reduce and reduce-scatter at even P), the hop
 * between them needs no signal, so a skip aimed at either of them skips the
 * block's notify to the next block.  (-1, -1) cancels a pending skip.
 */
int ring_debug_skip_notify(int rank, int step);

/*
 * Test hook for failure detection in the all-gather + GEMM: the next
 * ag_gemm, ag_gemm_kn or ag_gemm_ex launch on any thread copies the gather
 * piece that starts at A_g row `row` (a multiple of 16) but never publishes
 * its ready flag.  If those rows belong to another rank than the caller's,
 * the tiles that read them wait until the time bound, ring_status() (or
 * ring_status_ex() for a caller's workspace) reports RC_ERR_TIMEOUT, C is
 * undefined and the device stays usable; every role of the kernel stops
 * with no copy or MMA left in flight.  A row that starts no piece, or one of
 * the caller's own rows (read from its shard, never waited on), has no
 * effect.  -1 cancels a pending skip.  Errors: RC_ERR_INVALID (row < -1).
 */
int ag_gemm_debug_skip_piece(int row);

/*
 * Tracing hook: while dev_buf is set (a device buffer of `bytes` bytes), every
 * ring launch (the entry points listed for ring_debug_skip_notify) writes
 * three %globaltimer stamps (ns) per rank, slice and global step g, at word
 * (b*steps + g)*3 with b = (h*P + r)*slices + j for rank r, slice j and half
 * h (h = 0 except in the bidirectional reduce-scatter): the start of the
 * wait on the left neighbour, its end, and the end of the step (after the
 * notify).  steps = 2(P-1) for the all-reduce, P-1 otherwise.  Where two
 * ranks share a thread block (the all-reduce and reduce-scatter at even P),
 * the second rank's step waits on no other block: its wait starts and ends
 * when its step starts.  Rows whose stamps would not fit are not written.
 * NULL turns tracing off.  The caller owns the buffer and must keep it alive
 * while launches use it.
 */
int ring_debug_set_trace(void *dev_buf, size_t bytes);

/*
 * Measurement hook: the step-rate ceiling of the ring kernels.  Runs the
 * ring kernel's own streaming loop `reps` times over one range of `bytes`
 * bytes, in one launch of the ring's shape (8 blocks of 128 threads per SM,
 * block i taking the i-th equal share): add = 0 copies a to dst (an
 * all-gather step: one read and one write per byte); add = 1 stores the f32
 * sum a + b to dst (a reduce-scatter step: two reads and one write).  DEVICE
 * pointers, 256-byte aligned, bytes a multiple of 256, dst overlapping
 * neither input (RC_ERR_INVALID otherwise); 1 <= reps <= 100000.  With the
 * buffers small enough to stay in L2 (together well under its size), the
 * time of the launch gives the L2 rate that bounds a ring step whose data is
 * already on chip.  Not part of any collective.
 */
int ring_debug_l2_rate(void *dst, const void *a, const void *b, size_t bytes, int reps, int add, void *stream);

/* Frees the signal workspaces of all devices.  No call may be in flight. */
int ring_finalize(void);

/*
 * ring_allreduce_noalloc -- ring_allreduce for callers that cannot allocate
 * device memory.  The pages have no counterpart: this entry point exists
 * only because of how some callers run.
 *
 * ring_allreduce creates its signal workspace with cudaMalloc (and a
 * device-wide synchronisation) on the first call, and again whenever a larger
 * P needs a bigger one.  Some callers cannot allow that: a process whose
 * framework allocator already holds nearly all of the GPU's memory (so a
 * library cudaMalloc fails), code that must never trigger an allocation or an
 * implicit device synchronisation in its steady state, and runtimes that
 * forbid libraries from owning device allocations.  This variant keeps its
 * signal rows in a fixed array compiled into the library instead:
 * RC_NOALLOC_SCRATCH_BYTES bytes of device memory that every GPU which loads
 * the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Arguments, layout, validation and result: as ring_allreduce (the same
 * kernel runs with the same chunk segments; the result is bit-identical).
 * Additional limit: the signal rows of one call, slices*P*2(P-1)*P words plus
 * a 128-byte header, must fit in the array; the slice count is reduced to
 * fit (at P = 8 at most 73 slices, where ring_allreduce may use up to 152:
 * large calls then stream with fewer thread blocks and run slower), and P for
 * which even one slice does not fit (P > 32) is rejected with
 * RC_ERR_INVALID.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress and clears the array with
 * cudaMemsetAsync on `stream`; make that first call before any stream
 * capture.  Every call on a device shares the one array, which keeps the last
 * call's contents (signal rows hold epoch values, so nothing needs clearing
 * between calls).  Calls that overlap on the GPU -- on different streams
 * without ordering, or on different host threads -- race on the array and
 * give undefined results; issue them in stream order.  Errors raised by a
 * device wait are recorded in the array's header and read (and cleared) by
 * ring_status(), which allocates nothing either.
 */
#define RC_NOALLOC_SCRATCH_BYTES (256u * 1024u)
int ring_allreduce_noalloc(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* RINGCOLL_H */
