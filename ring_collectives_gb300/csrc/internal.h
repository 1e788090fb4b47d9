// internal.h -- declarations shared by the library's translation units
// (not part of the public ABI; the public header is include/ringcoll.h).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rc {

// Device-resident header at the start of a signal workspace (128 bytes).
struct WsHeader {
    uint32_t epoch;     // launches completed on this workspace; a launch signals with epoch+1
    uint32_t done;      // thread blocks of the running launch that have finished
    uint32_t status;    // 0, or the rc_status error code of the first failure
    uint32_t err_rank;  // where the first failure happened
    uint32_t err_step;
    uint32_t err_slice;
    uint32_t pad[26];   // pad[0]: abort word of the running launch; pad[1]: debug grid-barrier counter
};
static_assert(sizeof(WsHeader) == 128, "header is one 128-byte line");

enum RingMode { MODE_ALLREDUCE = 0, MODE_REDUCE_SCATTER = 1, MODE_ALL_GATHER = 2, MODE_RS_BIDIR = 3 };

// Arguments of one launch of the ring step engine.
struct RingParams {
    char *data;          // slots the ring runs on: bufs (all-reduce, reduce-scatter) or out (all-gather)
    size_t data_stride;  // bytes between slots
    const char *in;      // all-gather: input shards
    size_t in_stride;
    char *out;           // reduce-scatters: output chunks
    size_t out_stride;
    uint32_t *sig;       // signal rows, [S][P][rows][P] words
    WsHeader *hdr;
    size_t chunk;        // elements per chunk (all-gather: the shard length n)
    size_t chunk_stride; // elements between the starts of consecutive chunks of a slot (0: = chunk);
                         // larger when the launch runs one segment of every chunk
    int P, S, rows, mode;
    int discard;         // 1: drop the L2 lines of reduce-scatter partials once read (their data is dead)
    int segments;        // chunk segments run one after another (keeps a step's live data in L2)
    int ag_bulk;         // 1: all-gather copies move through shared memory with bulk (TMA) copies
    int debug_serial;    // 1: every step also waits for all blocks of the launch (debugging)
    int stagger_groups;  // > 1: slice j starts (j % stagger_groups) * stagger_ns later (phase-shifted rings)
    unsigned stagger_ns;
    int skip_rank, skip_step; // test hook: this rank skips its notify after this step (-1: none)
    int pair;            // 1: k_ring_pair (two ranks per thread block), else k_ring
    int hand_bytes;      // k_ring_pair: shared-memory bytes per block handed from rank r0 to r1 (multiple of 1024)
    unsigned long long timeout_ns;
    unsigned long long *trace; // optional step stamps (see ring_debug_set_trace); null: off
    size_t trace_words;
};

// Launch helpers implemented in ring_kernels.cu.  They return a cudaError_t.
cudaError_t launch_ring(const RingParams &p, int dtype, int threads, cudaStream_t st);
cudaError_t ring_max_coresident(int dtype, int threads, int device, int *blocks);
// ring_pair.cu: the same engine with two logical ranks per thread block.
cudaError_t launch_ring_pair(const RingParams &p, int dtype, cudaStream_t st);
cudaError_t ring_pair_max_coresident(int dtype, int device, int hand_bytes, int *blocks);
// fold_kernels.cu: order 0 = ring order (fused single-pass all-reduce), 1 = psum order.
cudaError_t launch_fold(char *data, size_t stride, int P, size_t N, size_t chunk, int dtype, int order, int sm_count,
                        cudaStream_t st);
cudaError_t launch_ppermute(const char *src, size_t src_stride, char *dst, size_t dst_stride, int P,
                            size_t n, int esize, int sm_count, cudaStream_t st);
// k_l2_rate: the ring's copy (add = 0) or f32 add (add = 1) loop, `reps` times over one range.
cudaError_t launch_l2_rate(char *dst, const char *a, const char *b, size_t bytes, int reps, int add, int sm_count,
                           cudaStream_t st);

// Host helpers implemented in api.cu and shared with ag_gemm.cu.
// set_error: records the calling thread's message; returns `code`.
int set_error(int code, const char *fmt, ...);
// prepare_workspace: the current device must be an sm_103 GPU with
// cooperative launch; grows the device's workspace to at least sig_words
// signal words and returns its header, words, SM count and wait bound.  The
// epoch in the header is shared by every launch that uses the workspace.
int prepare_workspace(size_t sig_words, WsHeader **hdr, uint32_t **sig, int *sm_count,
                      unsigned long long *timeout_ns);
// prepare_workspace_ext: the same with a caller-owned workspace (ext, ext_bytes
// bytes, 16-byte aligned, zeroed before first use); ext == nullptr takes the
// device's own.
int prepare_workspace_ext(void *ext, size_t ext_bytes, size_t sig_words, WsHeader **hdr, uint32_t **sig,
                          int *sm_count, unsigned long long *timeout_ns);

// Threads per block of the ring kernel, and the blocks per SM its register
// budget is sized for (build-time tuning knobs).
// Small blocks, many per SM: while some blocks wait on their left neighbour
// or drain a step, the others keep streaming (measured on GB300: 128 x 8 per
// SM beats 512 x 2 and 1024 x 1 by about 10 %).
#ifndef RC_RING_THREADS
#define RC_RING_THREADS 128
#endif
#ifndef RC_RING_MIN_BLOCKS
#define RC_RING_MIN_BLOCKS 8
#endif
// 32-byte vector pairs each thread keeps in flight in a reduce-scatter step.
// Measured on GB300 (P=8 x 64 MiB): 2 pairs at 8 blocks/SM 0.215 ms; 3 pairs
// 0.220; 4 pairs 0.225; 3-4 pairs at 6 blocks/SM 0.235-0.240; 64-thread
// blocks at 12-16 per SM 0.235-0.27.
#ifndef RC_RING_ADD_U
#define RC_RING_ADD_U 2
#endif
// Lines of the own input chunk prefetched into L2 while a standalone
// reduce-scatter round waits for its left neighbour (0: off).
#ifndef RC_RING_PREFETCH
#define RC_RING_PREFETCH 32
#endif
// Blocks per SM of the right-shift copy (256 threads each).  Measured on
// GB300 (P=8 x 64 MiB fp32): 1 -> 0.187 ms, 2 -> 0.178, 4 -> 0.182,
// 8 -> 0.167-0.169, 16 -> 0.169-0.170.
#ifndef RC_PPERMUTE_BLOCKS_PER_SM
#define RC_PPERMUTE_BLOCKS_PER_SM 8
#endif
constexpr int kRingThreads = RC_RING_THREADS;
// Threads per block and blocks per SM of k_ring_pair (two ranks per block,
// so the same thread count per SM as k_ring's 8 x 128).
#ifndef RC_PAIR_THREADS
#define RC_PAIR_THREADS 256
#endif
#ifndef RC_PAIR_MIN_BLOCKS
#define RC_PAIR_MIN_BLOCKS 4
#endif
constexpr int kPairThreads = RC_PAIR_THREADS;
// Slices start on multiples of this many elements (keeps 16-byte vectors aligned).
constexpr size_t kSliceGranule = 64;
// Bulk-copy staging of the ring's all-gather copies: stages x bytes of
// shared memory per block (build-time tuning knobs).  Measured on GB300 at
// P=8 x 64 MiB: 8 x 2 KiB beats 4 x 4 KiB and 2 x 8 KiB by 1-4 % and
// 4 x 2 KiB by 8 % (the copies are latency-bound on how far loads run
// ahead); 24 KiB per block (3 x 8 KiB, 6 x 4 KiB) is 20 % slower, and so is
// any staging depth once the largest shared-memory carveout is requested
// (0.254 ms): the launch needs the L1 share of the default carveout.
#ifndef RC_AG_STAGES
#define RC_AG_STAGES 8
#endif
#ifndef RC_AG_STAGE_BYTES
#define RC_AG_STAGE_BYTES 2048
#endif
constexpr int kAgStages = RC_AG_STAGES;
constexpr int kAgStageBytes = RC_AG_STAGE_BYTES;
static_assert(kAgStageBytes % 16 == 0 && kAgStages >= 2 && kAgStages <= 32, "bulk staging shape");

} // namespace rc
