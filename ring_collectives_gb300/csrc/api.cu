// api.cu -- the C ABI of libringcoll.so (declared in include/ringcoll.h):
// argument validation, the per-device signal workspace, launch-shape choice,
// device status read-back and error strings.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"
#include "ringcoll.h"

namespace {

thread_local std::string g_err;

// Unsigned value of environment variable `name`, or `dflt` when it is unset
// or malformed (initial values of the settings below; the setters override).
unsigned env_uint(const char *name, unsigned dflt)
{
    const char *e = getenv(name);
    if (!e || !*e) return dflt;
    char *end = nullptr;
    const unsigned long v = strtoul(e, &end, 10);
    return (end && *end == 0 && v <= 0xFFFFFFFFul) ? (unsigned)v : dflt;
}

std::atomic<unsigned> g_timeout_ms{env_uint("RC_TIMEOUT_MS", 2000)};   // ring_set_timeout_ms
std::atomic<int> g_slices{(int)env_uint("RC_SLICES", 0)};             // ring_set_slices
std::atomic<int> g_skip_rank{-1}, g_skip_step{-1};
std::atomic<unsigned long long *> g_trace{nullptr};
std::atomic<size_t> g_trace_words{0};
std::mutex g_mu;

constexpr int kMaxDevices = 64;
// One ring step touches a chunk of every rank.  When those P chunks exceed
// kL2NoSplitBytes, the chunks are split into segments run one after another,
// so the partial sums of a step stay in L2 until the next step reads them.
// Segment budgets measured on GB300 (126 MB L2; each segment adds 2(P-1)
// signal steps): up to 64 MiB of live chunks one pass is fastest; above it,
// k_ring runs best with 48 MiB segments (beating 32, 64 and 96 MiB by 1-7 %
// at P = 8, 16 and 32 with 16 MiB chunks), k_ring_pair -- which keeps the
// in-block hop's heads out of L2 -- with 64 MiB ones (P = 8 / 16 / 32:
// 24 MiB 0.515 / 2.15 / 9.14 ms, 32 MiB 0.436 / 1.87 / 7.74, 48 MiB
// 0.410 / 1.79 / 7.02, 64 MiB 0.388 / 1.70 / 6.57, 96 MiB 0.389 / 1.76 /
// 6.69).
constexpr size_t kDefaultL2LiveBytes = 48ull << 20;
constexpr size_t kPairL2LiveBytes = 64ull << 20;
constexpr size_t kL2NoSplitBytes = 64ull << 20;

// Tuning knob, read once from the environment: RC_L2_LIVE_BYTES (bytes; 0 =
// never segment); unset or malformed: the kernel's default above (returned
// as SIZE_MAX here).
size_t l2_live_bytes_setting()
{
    static const size_t v = [] {
        const char *e = getenv("RC_L2_LIVE_BYTES");
        if (!e || !*e) return SIZE_MAX;
        char *end = nullptr;
        const unsigned long long x = strtoull(e, &end, 10);
        return (end && *end == 0) ? (size_t)x : SIZE_MAX;
    }();
    return v;
}
// Phase-shifted slice rings.  The first step of a reduce-scatter reads two
// chunks from HBM per rank and is bound by HBM, while the later steps move
// data that is mostly in L2 and are bound by L2; when every slice ring runs
// in step, all of them are in the HBM-bound step at once.  Slice j therefore
// starts (j % G) * D later, G groups and D a fifth of the first step's time
// at ~6.5 TB/s (D in ns = its HBM bytes / 32500, capped at 50 us), so the
// groups' first steps overlap the others' L2-bound steps.  Measured on GB300
// (P=8 x 64 MiB fp32 all-reduce, D = 4.1 us): G=1 0.2150-0.2173 ms, G=2
// 0.2134-0.2143, G=3 0.2110-0.2119, G=4 0.2151-0.2154, G=5 0.2153-0.2160,
// G=6 0.2194-0.2201 (bf16: G=1 0.2152-0.2154, G=3 0.2123-0.2126).  The
// reduce-scatters use it too (P=8 x 64 MiB bf16: G=1 0.1356-0.1357 ms,
// G=2 0.1362-0.1364, G=3 0.1297-0.1300; bidirectional 0.1710-0.1715 ->
// 0.1697-0.1700 at G=3); the all-gather, whose first step is the own shard's
// copy, does not.  D as a seventh, a quarter or a third of the first step
// measured the same or slower (f32 0.2137-0.2139 / 0.2126-0.2139 /
// 0.2148 ms against 0.2130-0.2135; reduce-scatter 0.1307-0.1319 against
// 0.1298-0.1301).  Knob, read once: RC_RING_STAGGER = G (1 = off; unset or
// malformed = 3).
int stagger_groups_default()
{
    static const int v = [] {
        const char *e = getenv("RC_RING_STAGGER");
        if (!e || !*e) return 3;
        char *end = nullptr;
        const long x = strtol(e, &end, 10);
        return (end && *end == 0 && x >= 1 && x <= 16) ? (int)x : 3;
    }();
    return v;
}

void set_stagger(rc::RingParams &p, size_t es)
{
    p.stagger_groups = p.mode != rc::MODE_ALL_GATHER ? stagger_groups_default() : 1;
    const double first_step_bytes = 2.0 * p.P * ((double)p.chunk / (double)p.segments) * (double)es;
    const double ns = first_step_bytes / 32500.0;
    p.stagger_ns = p.stagger_groups > 1 ? (unsigned)(ns < 50000.0 ? ns : 50000.0) : 0u;
}

// Tuning knob, read once from the environment: RC_AG_BULK (1 = all-gather
// copies with bulk copies through shared memory, 0 = 32-byte vector loads
// and stores, for every collective; unset or malformed = the default per
// collective, see ag_bulk_for).
int ag_bulk_setting()
{
    static const int v = [] {
        const char *e = getenv("RC_AG_BULK");
        if (e && e[0] == '0' && e[1] == 0) return 0;
        if (e && e[0] == '1' && e[1] == 0) return 1;
        return -1;
    }();
    return v;
}

// All-gather steps of the all-reduce use vector copies, those of the
// standalone all-gather bulk copies.  Measured on GB300 (P=8 x 64 MiB fp32
// all-reduce with the phase-shifted rings): vector 0.2088-0.2091 ms, bulk
// 0.2104-0.2125 ms (before the stagger: bulk 0.2155 vs vector 0.2164).
int ag_bulk_for(int mode)
{
    const int v = ag_bulk_setting();
    return v >= 0 ? v : (mode == rc::MODE_ALL_GATHER ? 1 : 0);
}
// Two logical ranks per thread block (k_ring_pair) for the all-reduce and the
// reduce-scatter at even P; the hop inside a block hands the head of every
// slice over in shared memory.  Knobs, read once: RC_RING_PAIR=0 keeps k_ring
// (one rank per block) everywhere; RC_PAIR_SMEM = bytes handed over per block
// (a multiple of 1024; unset or malformed = the default below).
constexpr int kDefaultPairSmem = 44 << 10;
int pair_enabled()
{
    static const int v = env_uint("RC_RING_PAIR", 1) != 0;
    return v;
}
int pair_smem_bytes()
{
    static const int v = [] {
        const unsigned x = env_uint("RC_PAIR_SMEM", (unsigned)kDefaultPairSmem);
        return (x % 1024 == 0 && x <= (160u << 10)) ? (int)x : kDefaultPairSmem;
    }();
    return v;
}

// Debug knob, read once from the environment: RC_DEBUG_SERIAL=1 makes every
// step of a ring launch also wait for all blocks of the launch (a bounded
// grid barrier), ruling fine-grained synchronisation in or out as the cause
// of a wrong result.
int debug_serial()
{
    static const int v = env_uint("RC_DEBUG_SERIAL", 0) != 0;
    return v;
}
constexpr size_t kMinSliceBytes = 32 << 10; // a slice below this is not worth its own ring
constexpr uint64_t kEpochResetAt = 1ull << 30; // re-zero the workspace long before 32-bit wrap

struct DeviceState {
    bool probed = false;
    int supported = 0;  // 1 if sm_103 and cooperative launch are available
    int sm_count = 0;
    int max_blocks[3] = {0, 0, 0}; // co-resident ring blocks per dtype
    int pair_blocks[3] = {0, 0, 0}; // co-resident k_ring_pair blocks per dtype (0: pair kernel unavailable)
    void *ws = nullptr;  // WsHeader followed by the signal words
    size_t ws_bytes = 0;
    uint64_t launches = 0;
};
DeviceState g_dev[kMaxDevices];

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(RC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t elem_size(int dtype)
{
    switch (dtype) {
    case RC_F32: return 4;
    case RC_BF16: return 2;
    case RC_I32: return 4;
    default: return 0;
    }
}

// Element accesses need element-aligned slots: base and stride multiples of the element size.
bool elem_aligned(const void *base, size_t stride, size_t es)
{
    return ((uintptr_t)base % es) == 0 && (stride % es) == 0;
}

// [lo, hi) byte range spanned by P slots of `bytes` each.
bool regions_overlap(const void *a, size_t a_stride, size_t a_bytes, const void *b, size_t b_stride,
                     size_t b_bytes, int P)
{
    const uintptr_t a0 = (uintptr_t)a, a1 = a0 + (size_t)(P - 1) * a_stride + a_bytes;
    const uintptr_t b0 = (uintptr_t)b, b1 = b0 + (size_t)(P - 1) * b_stride + b_bytes;
    return a0 < b1 && b0 < a1;
}

// Current device, probed once: compute capability 10.3 and cooperative launch.
int current_device(int *dev_out, DeviceState **st_out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RC_ERR_UNSUPPORTED, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(RC_ERR_UNSUPPORTED, "device index %d out of range", dev);
    DeviceState &st = g_dev[dev];
    if (!st.probed) {
        int major = 0, minor = 0, coop = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
        st.supported = (major == 10 && minor == 3 && coop) ? 1 : 0;
        if (st.supported) {
            for (int dt = 0; dt < 3; ++dt) {
                e = rc::ring_max_coresident(dt, rc::kRingThreads, dev, &st.max_blocks[dt]);
                if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
                if (pair_enabled()) {
                    // Without a usable launch shape for the two-rank kernel
                    // (e.g. a shared-memory setting this device cannot grant)
                    // every ring collective runs on k_ring instead.
                    e = rc::ring_pair_max_coresident(dt, dev, pair_smem_bytes(), &st.pair_blocks[dt]);
                    if (e != cudaSuccess) {
                        (void)cudaGetLastError();
                        st.pair_blocks[dt] = 0;
                    }
                }
            }
        }
        st.probed = true;
        if (!st.supported)
            return fail(RC_ERR_UNSUPPORTED, "device %d is sm_%d%d (cooperative launch %d); this library is built "
                        "for sm_103a", dev, major, minor, coop);
    }
    if (!st.supported) return fail(RC_ERR_UNSUPPORTED, "device %d is not an sm_103 GPU", dev);
    *dev_out = dev;
    *st_out = &st;
    return RC_OK;
}

// Makes the workspace at least `sig_bytes` of signal words (after the header).
int ensure_workspace(DeviceState &st, size_t sig_bytes)
{
    const size_t need = sizeof(rc::WsHeader) + sig_bytes;
    cudaError_t e;
    if (st.ws && (st.ws_bytes < need || st.launches >= kEpochResetAt)) {
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "synchronise before workspace resize");
        if (st.ws_bytes < need) {
            cudaFree(st.ws);
            st.ws = nullptr;
            st.ws_bytes = 0;
        } else {
            e = cudaMemset(st.ws, 0, st.ws_bytes);
            if (e == cudaSuccess) e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return cuda_fail(e, "workspace reset");
            st.launches = 0;
        }
    }
    if (!st.ws) {
        size_t bytes = (need + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
        e = cudaMalloc(&st.ws, bytes);
        if (e != cudaSuccess) {
            st.ws = nullptr;
            return fail(RC_ERR_NOMEM, "signal workspace of %zu bytes: %s", bytes, cudaGetErrorString(e));
        }
        e = cudaMemset(st.ws, 0, bytes);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "workspace zeroing");
        st.ws_bytes = bytes;
        st.launches = 0;
    }
    return RC_OK;
}

// Slices per rank for a chunk of chunk_bytes (see ring_set_slices).
// blocks: co-resident blocks of the kernel; per_slice: its blocks per slice ring.
int choose_slices(int blocks, int per_slice, size_t chunk_elems, size_t chunk_bytes, int *S_out)
{
    const int cap = blocks / per_slice;
    if (cap < 1)
        return fail(RC_ERR_UNSUPPORTED, "%d blocks per slice exceed the %d co-resident blocks of this device",
                    per_slice, blocks);
    long S;
    const int user = g_slices.load();
    if (user > 0) {
        S = user;
    } else {
        S = cap; // every co-resident block slot of the GPU holds one (rank, slice)
        const long by_size = (long)(chunk_bytes / kMinSliceBytes);
        if (S > by_size) S = by_size;
    }
    const long by_granule = (long)(chunk_elems / rc::kSliceGranule);
    if (S > by_granule) S = by_granule;
    if (S > cap) S = cap;
    if (S < 1) S = 1;
    *S_out = (int)S;
    return RC_OK;
}

// k_ring_pair takes the all-reduce and both reduce-scatters at even P when
// every slice starts on a 32-byte boundary (slot bases, strides, chunk starts
// and, for the bidirectional one, the second half of every chunk multiples of
// 32 bytes) and the all-gather steps use vector copies.
bool pair_fits(const rc::RingParams &p, const DeviceState &st, int dtype, size_t es)
{
    if (!pair_enabled() || st.pair_blocks[dtype] < 1) return false;
    if (p.mode == rc::MODE_ALL_GATHER) return false;
    if (p.P < 2 || (p.P & 1) || p.ag_bulk) return false;
    const size_t cs = p.chunk_stride ? p.chunk_stride : p.chunk;
    if (((uintptr_t)p.data | p.data_stride | (cs * es)) & 31u) return false;
    if (p.mode != rc::MODE_ALLREDUCE && (((uintptr_t)p.out | p.out_stride) & 31u)) return false;
    if (p.mode == rc::MODE_RS_BIDIR && ((p.chunk / 2) * es) & 31u) return false;
    return true;
}

// Chooses the kernel, slices and segments of a ring launch (the same for every
// workspace).  allow_pair = 0 plans k_ring even where k_ring_pair would run.
int plan_ring(rc::RingParams &p, int dtype, DeviceState *st, int allow_pair = 1)
{
    int rc_ = RC_OK;
    const size_t es = elem_size(dtype);
    p.ag_bulk = ag_bulk_for(p.mode);
    p.pair = allow_pair && pair_fits(p, *st, dtype, es) ? 1 : 0;
    p.hand_bytes = p.pair ? pair_smem_bytes() : 0;
    // The bidirectional reduce-scatter runs two rings (top and bottom halves) per slice.
    const int rings = p.mode == rc::MODE_RS_BIDIR ? 2 : 1;
    const size_t ring_elems = p.chunk / (size_t)rings;
    if (p.pair)
        rc_ = choose_slices(st->pair_blocks[dtype], p.P / 2 * rings, ring_elems, ring_elems * es, &p.S);
    else
        rc_ = choose_slices(st->max_blocks[dtype], p.P * rings, ring_elems, ring_elems * es, &p.S);
    if (rc_) return rc_;
    {
        const size_t setting = l2_live_bytes_setting();
        const size_t dflt = p.pair ? kPairL2LiveBytes : kDefaultL2LiveBytes;
        const size_t live = (size_t)p.P * p.chunk * es, budget = setting == SIZE_MAX ? dflt : setting;
        const bool split = budget && (live > kL2NoSplitBytes || budget < kDefaultL2LiveBytes);
        size_t G = split ? (live + budget - 1) / budget : 1;
        const size_t max_g = ring_elems / ((size_t)p.S * rc::kSliceGranule); // keep every slice non-empty
        if (G > max_g) G = max_g;
        if (G > 64) G = 64;
        if (G < 1) G = 1;
        p.segments = (int)G;
    }
    if (p.chunk_stride == 0) p.chunk_stride = p.chunk;
    set_stagger(p, es);
    return rc_;
}

size_t ring_sig_bytes(const rc::RingParams &p) { return (size_t)p.S * p.P * (size_t)p.rows * p.P * 4; }

// Workspace bytes a caller must provide for a ring launch of these
// parameters: the larger of the two kernels' signal rows (which kernel runs
// depends on the caller's slot alignment), plus the header; 0 when no
// supported device is current.
size_t ring_ws_bytes_for(rc::RingParams p, int dtype)
{
    int dev;
    DeviceState *st = nullptr;
    if (current_device(&dev, &st)) return 0;
    // placeholder slots on 32-byte boundaries, so the pair kernel is planned
    // wherever the caller's layout could let it run
    p.data_stride = (p.data_stride + 31) & ~(size_t)31;
    p.out_stride = (p.out_stride + 31) & ~(size_t)31;
    rc::RingParams a = p, b = p;
    if (plan_ring(a, dtype, st, 1) || plan_ring(b, dtype, st, 0)) return 0;
    const size_t x = ring_sig_bytes(a), y = ring_sig_bytes(b);
    return sizeof(rc::WsHeader) + (x > y ? x : y);
}

// Launches a planned ring collective.  ext_ws == nullptr: the device's own
// workspace; otherwise the caller's (ext_bytes long, zeroed before first use).
int run_ring(rc::RingParams &p, int dtype, cudaStream_t st_cuda, void *ext_ws = nullptr, size_t ext_bytes = 0)
{
    int dev;
    DeviceState *st = nullptr;
    int rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    rc_ = plan_ring(p, dtype, st);
    if (rc_) return rc_;
    const size_t sig_bytes = ring_sig_bytes(p);
    std::unique_lock<std::mutex> lock(g_mu, std::defer_lock);
    if (ext_ws) {
        if (ext_bytes < sizeof(rc::WsHeader) + sig_bytes)
            return fail(RC_ERR_INVALID, "workspace of %zu bytes is below the %zu this call needs", ext_bytes,
                        sizeof(rc::WsHeader) + sig_bytes);
        if ((uintptr_t)ext_ws & 15u) return fail(RC_ERR_INVALID, "workspace must be 16-byte aligned");
        p.hdr = (rc::WsHeader *)ext_ws;
        p.sig = (uint32_t *)((char *)ext_ws + sizeof(rc::WsHeader));
    } else {
        lock.lock();
        rc_ = ensure_workspace(*st, sig_bytes);
        if (rc_) return rc_;
        p.hdr = (rc::WsHeader *)st->ws;
        p.sig = (uint32_t *)((char *)st->ws + sizeof(rc::WsHeader));
    }
    p.timeout_ns = (unsigned long long)g_timeout_ms.load() * 1000000ull;
    p.skip_rank = g_skip_rank.exchange(-1);
    p.skip_step = g_skip_step.exchange(-1);
    p.trace = g_trace.load();
    p.trace_words = g_trace_words.load();
    p.debug_serial = debug_serial();
    cudaError_t e = p.pair ? rc::launch_ring_pair(p, dtype, st_cuda) : rc::launch_ring(p, dtype, rc::kRingThreads, st_cuda);
    if (e != cudaSuccess) return cuda_fail(e, "ring kernel launch");
    if (!ext_ws) st->launches += (uint64_t)p.segments; // the launch advances the epoch by its segment count
    return RC_OK;
}

int run_copy(const void *src, size_t src_stride, void *dst, size_t dst_stride, int P, size_t n, int dtype,
             cudaStream_t s)
{
    int dev;
    DeviceState *st = nullptr;
    int rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    const size_t es = elem_size(dtype);
    cudaError_t e = rc::launch_ppermute((const char *)src, src_stride, (char *)dst, dst_stride, P, n, (int)es,
                                        st->sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "copy kernel launch");
    return RC_OK;
}

} // namespace

namespace rc {

int set_error(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int prepare_workspace(size_t sig_words, WsHeader **hdr, uint32_t **sig, int *sm_count,
                      unsigned long long *timeout_ns)
{
    int dev;
    DeviceState *st = nullptr;
    int rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    std::lock_guard<std::mutex> lock(g_mu);
    rc_ = ensure_workspace(*st, sig_words * 4);
    if (rc_) return rc_;
    *hdr = (WsHeader *)st->ws;
    *sig = (uint32_t *)((char *)st->ws + sizeof(WsHeader));
    *sm_count = st->sm_count;
    *timeout_ns = (unsigned long long)g_timeout_ms.load() * 1000000ull;
    st->launches++;
    return RC_OK;
}

int prepare_workspace_ext(void *ext, size_t ext_bytes, size_t sig_words, WsHeader **hdr, uint32_t **sig,
                          int *sm_count, unsigned long long *timeout_ns)
{
    if (!ext) return prepare_workspace(sig_words, hdr, sig, sm_count, timeout_ns);
    int dev;
    DeviceState *st = nullptr;
    int rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    const size_t need = sizeof(WsHeader) + sig_words * 4;
    if ((uintptr_t)ext & 15u) return fail(RC_ERR_INVALID, "workspace must be 16-byte aligned");
    if (ext_bytes < need)
        return fail(RC_ERR_INVALID, "workspace of %zu bytes is below the %zu this call needs", ext_bytes, need);
    *hdr = (WsHeader *)ext;
    *sig = (uint32_t *)((char *)ext + sizeof(WsHeader));
    *sm_count = st->sm_count;
    *timeout_ns = (unsigned long long)g_timeout_ms.load() * 1000000ull;
    return RC_OK;
}

} // namespace rc

extern "C" {

const char *ring_last_error(void) { return g_err.c_str(); }

int ring_set_timeout_ms(unsigned ms)
{
    if (ms < 1 || ms > 600000) return fail(RC_ERR_INVALID, "timeout %u ms outside 1..600000", ms);
    g_timeout_ms.store(ms);
    return RC_OK;
}

int ring_set_slices(int slices)
{
    if (slices < 0 || slices > 4096) return fail(RC_ERR_INVALID, "slices %d outside 0..4096", slices);
    g_slices.store(slices);
    return RC_OK;
}

int ring_debug_skip_notify(int rank, int step)
{
    if (rank < -1 || step < -1) return fail(RC_ERR_INVALID, "bad skip_notify arguments");
    g_skip_rank.store(rank);
    g_skip_step.store(step);
    return RC_OK;
}

int ring_debug_l2_rate(void *dst, const void *a, const void *b, size_t bytes, int reps, int add, void *stream)
{
    if (!dst || !a || (add && !b)) return fail(RC_ERR_INVALID, "null pointer");
    if (reps < 1 || reps > 100000) return fail(RC_ERR_INVALID, "reps %d outside 1..100000", reps);
    if (bytes % 256 || ((uintptr_t)dst | (uintptr_t)a | (uintptr_t)(add ? b : a)) % 256)
        return fail(RC_ERR_INVALID, "pointers and size must be multiples of 256 bytes");
    if (regions_overlap(dst, 0, bytes, a, 0, bytes, 1) || (add && regions_overlap(dst, 0, bytes, b, 0, bytes, 1)))
        return fail(RC_ERR_INVALID, "dst overlaps an input");
    if (bytes == 0) return RC_OK;
    int dev;
    DeviceState *st = nullptr;
    int rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    cudaError_t e = rc::launch_l2_rate((char *)dst, (const char *)a, (const char *)b, bytes, reps, add ? 1 : 0,
                                       st->sm_count, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "probe kernel launch");
    return RC_OK;
}

int ring_debug_set_trace(void *dev_buf, size_t bytes)
{
    if (!dev_buf) bytes = 0;
    g_trace_words.store(bytes / 8);
    g_trace.store((unsigned long long *)dev_buf);
    return RC_OK;
}

int ring_ppermute_right(const void *src_base, size_t src_stride, void *dst_base, size_t dst_stride, int P,
                        size_t n, int dtype, void *stream)
{
    const size_t es = elem_size(dtype);
    if (!es) return fail(RC_ERR_INVALID, "unknown dtype %d", dtype);
    if (P < 1 || P > RC_MAX_P) return fail(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (n == 0) return RC_OK;
    if (!src_base || !dst_base) return fail(RC_ERR_INVALID, "null slot base");
    if (P > 1 && (src_stride < n * es || dst_stride < n * es))
        return fail(RC_ERR_INVALID, "stride below the %zu bytes of a slot", n * es);
    if (regions_overlap(src_base, src_stride, n * es, dst_base, dst_stride, n * es, P))
        return fail(RC_ERR_INVALID, "src and dst slots overlap");
    if (!elem_aligned(src_base, src_stride, es) || !elem_aligned(dst_base, dst_stride, es))
        return fail(RC_ERR_INVALID, "slot bases and strides must be multiples of the %zu-byte element", es);
    return run_copy(src_base, src_stride, dst_base, dst_stride, P, n, dtype, (cudaStream_t)stream);
}

// Validation and launch parameters of the ring collectives.  Results:
// RC_OK (p filled), kNothing (no work), kCopy (P = 1: a plain copy), or an
// error code (message set).
constexpr int kNothing = -1, kCopy = -2;

static int ag_params(const void *in_base, size_t in_stride, void *out_base, size_t out_stride, int P, size_t n,
                     int dtype, rc::RingParams &p)
{
    const size_t es = elem_size(dtype);
    if (!es) return fail(RC_ERR_INVALID, "unknown dtype %d", dtype);
    if (P < 1 || P > RC_MAX_P) return fail(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (n == 0) return kNothing;
    if (!in_base || !out_base) return fail(RC_ERR_INVALID, "null slot base");
    if (P > 1 && (in_stride < n * es || out_stride < (size_t)P * n * es))
        return fail(RC_ERR_INVALID, "stride below a slot's bytes (in %zu, out %zu)", n * es, (size_t)P * n * es);
    if (regions_overlap(in_base, in_stride, n * es, out_base, out_stride, (size_t)P * n * es, P))
        return fail(RC_ERR_INVALID, "in and out slots overlap");
    if (!elem_aligned(in_base, in_stride, es) || !elem_aligned(out_base, out_stride, es))
        return fail(RC_ERR_INVALID, "slot bases and strides must be multiples of the %zu-byte element", es);
    if (P == 1) return kCopy;
    p = rc::RingParams{};
    p.data = (char *)out_base;
    p.data_stride = out_stride;
    p.in = (const char *)in_base;
    p.in_stride = in_stride;
    p.chunk = n;
    p.P = P;
    p.rows = P - 1;
    p.mode = rc::MODE_ALL_GATHER;
    p.discard = 0;
    return RC_OK;
}

static int all_gather_run(const void *in_base, size_t in_stride, void *out_base, size_t out_stride, int P, size_t n,
                          int dtype, void *ws, size_t ws_bytes, void *stream)
{
    rc::RingParams p;
    const int v = ag_params(in_base, in_stride, out_base, out_stride, P, n, dtype, p);
    if (v == kNothing) return RC_OK;
    if (v == kCopy) return run_copy(in_base, in_stride, out_base, out_stride, 1, n, dtype, (cudaStream_t)stream);
    if (v) return v;
    return run_ring(p, dtype, (cudaStream_t)stream, ws, ws_bytes);
}

int ring_all_gather(const void *in_base, size_t in_stride, void *out_base, size_t out_stride, int P, size_t n,
                    int dtype, void *stream)
{
    return all_gather_run(in_base, in_stride, out_base, out_stride, P, n, dtype, nullptr, 0, stream);
}

int ring_all_gather_ex(const void *in_base, size_t in_stride, void *out_base, size_t out_stride, int P, size_t n,
                       int dtype, void *workspace, size_t ws_bytes, void *stream)
{
    if (!workspace) return fail(RC_ERR_INVALID, "null workspace");
    return all_gather_run(in_base, in_stride, out_base, out_stride, P, n, dtype, workspace, ws_bytes, stream);
}

size_t ring_all_gather_workspace_bytes(int P, size_t n, int dtype)
{
    rc::RingParams p;
    const size_t es = elem_size(dtype);
    const int v = ag_params((const void *)(uintptr_t)4096, n * es, (void *)((uintptr_t)1 << 40), (size_t)P * n * es,
                            P, n, dtype, p);
    if (v == kNothing || v == kCopy) return sizeof(rc::WsHeader);
    if (v) return 0;
    return ring_ws_bytes_for(p, dtype);
}

// mode: MODE_REDUCE_SCATTER or MODE_RS_BIDIR.
static int rs_params(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P, size_t N,
                     int dtype, int mode, rc::RingParams &p)
{
    const size_t es = elem_size(dtype);
    if (!es) return fail(RC_ERR_INVALID, "unknown dtype %d", dtype);
    if (P < 1 || P > RC_MAX_P) return fail(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (N % (size_t)P) return fail(RC_ERR_INVALID, "N=%zu is not a multiple of P=%d", N, P);
    if (N == 0) return kNothing;
    if (!bufs_base || !out_base) return fail(RC_ERR_INVALID, "null slot base");
    const size_t c = N / (size_t)P;
    if (P > 1 && (bufs_stride < N * es || out_stride < c * es))
        return fail(RC_ERR_INVALID, "stride below a slot's bytes (bufs %zu, out %zu)", N * es, c * es);
    if (regions_overlap(bufs_base, bufs_stride, N * es, out_base, out_stride, c * es, P))
        return fail(RC_ERR_INVALID, "bufs and out slots overlap");
    if (!elem_aligned(bufs_base, bufs_stride, es) || !elem_aligned(out_base, out_stride, es))
        return fail(RC_ERR_INVALID, "slot bases and strides must be multiples of the %zu-byte element", es);
    if (P == 1) return kCopy;
    p = rc::RingParams{};
    p.data = (char *)bufs_base;
    p.data_stride = bufs_stride;
    p.out = (char *)out_base;
    p.out_stride = out_stride;
    p.chunk = c;
    p.P = P;
    p.rows = mode == rc::MODE_RS_BIDIR ? 2 * (P - 1) : P - 1;   // bidirectional: P-1 steps per half
    p.mode = mode;
    p.discard = 1;
    return RC_OK;
}

static int rs_run(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P, size_t N, int dtype,
                  int mode, void *ws, size_t ws_bytes, void *stream)
{
    rc::RingParams p;
    const int v = rs_params(bufs_base, bufs_stride, out_base, out_stride, P, N, dtype, mode, p);
    if (v == kNothing) return RC_OK;
    if (v == kCopy) return run_copy(bufs_base, bufs_stride, out_base, out_stride, 1, N, dtype, (cudaStream_t)stream);
    if (v) return v;
    return run_ring(p, dtype, (cudaStream_t)stream, ws, ws_bytes);
}

static size_t rs_ws_bytes(int P, size_t N, int dtype, int mode)
{
    rc::RingParams p;
    const size_t es = elem_size(dtype);
    const int v = rs_params((void *)(uintptr_t)4096, N * es, (void *)((uintptr_t)1 << 40), (P > 0 ? N / (size_t)P : 0) * es,
                            P, N, dtype, mode, p);
    if (v == kNothing || v == kCopy) return sizeof(rc::WsHeader);
    if (v) return 0;
    return ring_ws_bytes_for(p, dtype);
}

int ring_reduce_scatter(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P, size_t N,
                        int dtype, void *stream)
{
    return rs_run(bufs_base, bufs_stride, out_base, out_stride, P, N, dtype, rc::MODE_REDUCE_SCATTER, nullptr, 0,
                  stream);
}

int ring_reduce_scatter_ex(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P, size_t N,
                           int dtype, void *workspace, size_t ws_bytes, void *stream)
{
    if (!workspace) return fail(RC_ERR_INVALID, "null workspace");
    return rs_run(bufs_base, bufs_stride, out_base, out_stride, P, N, dtype, rc::MODE_REDUCE_SCATTER, workspace,
                  ws_bytes, stream);
}

size_t ring_reduce_scatter_workspace_bytes(int P, size_t N, int dtype)
{
    return rs_ws_bytes(P, N, dtype, rc::MODE_REDUCE_SCATTER);
}

int ring_reduce_scatter_bidir(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P,
                              size_t N, int dtype, void *stream)
{
    return rs_run(bufs_base, bufs_stride, out_base, out_stride, P, N, dtype, rc::MODE_RS_BIDIR, nullptr, 0, stream);
}

int ring_reduce_scatter_bidir_ex(void *bufs_base, size_t bufs_stride, void *out_base, size_t out_stride, int P,
                                 size_t N, int dtype, void *workspace, size_t ws_bytes, void *stream)
{
    if (!workspace) return fail(RC_ERR_INVALID, "null workspace");
    return rs_run(bufs_base, bufs_stride, out_base, out_stride, P, N, dtype, rc::MODE_RS_BIDIR, workspace, ws_bytes,
                  stream);
}

size_t ring_reduce_scatter_bidir_workspace_bytes(int P, size_t N, int dtype)
{
    return rs_ws_bytes(P, N, dtype, rc::MODE_RS_BIDIR);
}

int ring_allreduce(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *stream)
{
    const size_t es = elem_size(dtype);
    if (!es) return fail(RC_ERR_INVALID, "unknown dtype %d", dtype);
    if (P < 1 || P > RC_MAX_P) return fail(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (N % (size_t)P) return fail(RC_ERR_INVALID, "N=%zu is not a multiple of P=%d", N, P);
    if (N == 0 || P == 1) return RC_OK;
    if (!bufs_base) return fail(RC_ERR_INVALID, "null slot base");
    if (stride < N * es) return fail(RC_ERR_INVALID, "stride %zu below the %zu bytes of a slot", stride, N * es);
    if (!elem_aligned(bufs_base, stride, es))
        return fail(RC_ERR_INVALID, "slot base and stride must be multiples of the %zu-byte element", es);
    const size_t c = N / (size_t)P;
    rc::RingParams p{};
    p.data = (char *)bufs_base;
    p.data_stride = stride;
    p.chunk = c;
    p.P = P;
    p.rows = 2 * (P - 1);
    p.mode = rc::MODE_ALLREDUCE;
    p.discard = 1;
    return run_ring(p, dtype, (cudaStream_t)stream);
}

static int run_fold(void *bufs_base, size_t stride, int P, size_t N, int dtype, int order, void *stream)
{
    const size_t es = elem_size(dtype);
    if (!es) return fail(RC_ERR_INVALID, "unknown dtype %d", dtype);
    if (P < 1 || P > RC_MAX_P) return fail(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (order == 0 && N % (size_t)P) return fail(RC_ERR_INVALID, "N=%zu is not a multiple of P=%d", N, P);
    if (N == 0 || (P == 1 && order == 0)) return RC_OK;
    if (!bufs_base) return fail(RC_ERR_INVALID, "null slot base");
    if (P > 1 && stride < N * es) return fail(RC_ERR_INVALID, "stride %zu below the %zu bytes of a slot", stride, N * es);
    if (!elem_aligned(bufs_base, stride, es))
        return fail(RC_ERR_INVALID, "slot base and stride must be multiples of the %zu-byte element", es);
    int dev;
    DeviceState *st = nullptr;
    int rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    cudaError_t e = rc::launch_fold((char *)bufs_base, P > 1 ? stride : N * es, P, N, order == 0 ? N / (size_t)P : 1,
                                    dtype, order, st->sm_count, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "fold kernel launch");
    return RC_OK;
}

int ring_allreduce_fused(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *stream)
{
    return run_fold(bufs_base, stride, P, N, dtype, 0, stream);
}

int ring_psum(void *bufs_base, size_t stride, int P, size_t n, int dtype, void *stream)
{
    return run_fold(bufs_base, stride, P, n, dtype, 1, stream);
}

// Validation and parameters shared by ring_allreduce and ring_allreduce_ex.
static int allreduce_params(void *bufs_base, size_t stride, int P, size_t N, int dtype, rc::RingParams &p)
{
    const size_t es = elem_size(dtype);
    if (!es) return fail(RC_ERR_INVALID, "unknown dtype %d", dtype);
    if (P < 1 || P > RC_MAX_P) return fail(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (N % (size_t)P) return fail(RC_ERR_INVALID, "N=%zu is not a multiple of P=%d", N, P);
    if (N == 0 || P == 1) return -1; // nothing to do
    if (!bufs_base) return fail(RC_ERR_INVALID, "null slot base");
    if (stride < N * es) return fail(RC_ERR_INVALID, "stride %zu below the %zu bytes of a slot", stride, N * es);
    if (!elem_aligned(bufs_base, stride, es))
        return fail(RC_ERR_INVALID, "slot base and stride must be multiples of the %zu-byte element", es);
    p = rc::RingParams{};
    p.data = (char *)bufs_base;
    p.data_stride = stride;
    p.chunk = N / (size_t)P;
    p.P = P;
    p.rows = 2 * (P - 1);
    p.mode = rc::MODE_ALLREDUCE;
    p.discard = 1;
    return RC_OK;
}

size_t ring_allreduce_workspace_bytes(int P, size_t N, int dtype)
{
    rc::RingParams p;
    int v = allreduce_params((void *)(uintptr_t)4096, N * elem_size(dtype), P, N, dtype, p);
    if (v < 0) return sizeof(rc::WsHeader);
    if (v) return 0;
    return ring_ws_bytes_for(p, dtype);
}

int ring_allreduce_ex(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *workspace, size_t ws_bytes,
                      void *stream)
{
    rc::RingParams p;
    int v = allreduce_params(bufs_base, stride, P, N, dtype, p);
    if (v < 0) return RC_OK;
    if (v) return v;
    if (!workspace) return fail(RC_ERR_INVALID, "null workspace");
    return run_ring(p, dtype, (cudaStream_t)stream, workspace, ws_bytes);
}

// Host all-reduce: above kHostPipeMinBytes of slots the copies and the ring
// run in segments (segment q = the same sub-range of every chunk, so every
// element keeps its chunk and its fold order): host-to-device copies on one
// internal stream, the ring launches on the caller's stream, device-to-host
// copies on a second internal stream, ordered by events, so both copy
// directions and the kernels overlap.
// Measured on GB300 (P=8 x 64 MiB fp32): one pass 5.54 ms; segments of
// 16-32 MiB 3.63 ms, 64 MiB 3.55 ms, 128 MiB 3.86 ms.  The host link moves
// ~210 GB/s in and ~193 GB/s out alone, ~171 GB/s each way together.
constexpr size_t kHostPipeMinBytes = 128ull << 20;
constexpr size_t kHostPipeSegmentBytes = 64ull << 20;

// Tuning knob, read once from the environment: RC_HOST_SEGMENT_BYTES (bytes of
// all slots per segment of the host all-reduce; unset or malformed = the
// default above; 0 = no segments).
static size_t host_segment_bytes()
{
    static const size_t v = [] {
        const char *e = getenv("RC_HOST_SEGMENT_BYTES");
        if (!e || !*e) return kHostPipeSegmentBytes;
        char *end = nullptr;
        const unsigned long long x = strtoull(e, &end, 10);
        return (end && *end == 0) ? (size_t)x : kHostPipeSegmentBytes;
    }();
    return v;
}

struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
};
HostPipe g_pipe[kMaxDevices];

static int host_pipe_streams(int dev, HostPipe **out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    HostPipe &hp = g_pipe[dev];
    if (!hp.in) {
        cudaError_t e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            if (hp.in) cudaStreamDestroy(hp.in);
            hp.in = hp.out = nullptr;
            return cuda_fail(e, "copy stream creation");
        }
    }
    *out = &hp;
    return RC_OK;
}

// Elements [lo, lo+n) of every chunk (chunks c elements apart) of all P
// slots: one pitched copy of P*P rows when both sides hold the slots back to
// back (slot r, chunk k is row r*P+k of a [P*P][c] matrix), else one pitched
// copy of P rows per slot.
static cudaError_t copy_segment(void *dst, size_t dst_stride, const void *src, size_t src_stride, int P, size_t c,
                                size_t lo, size_t n, size_t es, cudaMemcpyKind kind, cudaStream_t s)
{
    const size_t row = (size_t)P * c * es;
    if (dst_stride == row && src_stride == row)
        return cudaMemcpy2DAsync((char *)dst + lo * es, c * es, (const char *)src + lo * es, c * es, n * es,
                                 (size_t)P * (size_t)P, kind, s);
    for (int r = 0; r < P; ++r) {
        cudaError_t e = cudaMemcpy2DAsync((char *)dst + (size_t)r * dst_stride + lo * es, c * es,
                                          (const char *)src + (size_t)r * src_stride + lo * es, c * es, n * es,
                                          (size_t)P, kind, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int ring_allreduce_host(const void *h_in, size_t h_in_stride, void *h_out, size_t h_out_stride, void *d_bufs,
                        size_t d_stride, int P, size_t N, int dtype, void *stream)
{
    const size_t es = elem_size(dtype);
    if (!es) return fail(RC_ERR_INVALID, "unknown dtype %d", dtype);
    if (P < 1 || P > RC_MAX_P) return fail(RC_ERR_INVALID, "P=%d outside 1..%d", P, RC_MAX_P);
    if (N % (size_t)P) return fail(RC_ERR_INVALID, "N=%zu is not a multiple of P=%d", N, P);
    if (N == 0) return RC_OK;
    if (!h_in || !h_out || !d_bufs) return fail(RC_ERR_INVALID, "null pointer");
    const size_t row = N * es;
    if ((P > 1 && (h_in_stride < row || h_out_stride < row || d_stride < row)))
        return fail(RC_ERR_INVALID, "stride below the %zu bytes of a slot", row);
    if (P == 1) h_in_stride = h_out_stride = d_stride = row;
    if (!elem_aligned(d_bufs, d_stride, es))
        return fail(RC_ERR_INVALID, "device slot base and stride must be multiples of the %zu-byte element", es);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t c = N / (size_t)P;
    const size_t total = (size_t)P * row;
    const size_t seg_bytes = host_segment_bytes();
    size_t G = total >= kHostPipeMinBytes && P > 1 && seg_bytes ? total / seg_bytes : 1;
    if (G > 64) G = 64;
    if (G > c / (4 * rc::kSliceGranule)) G = c / (4 * rc::kSliceGranule);
    if (G < 2) {
        cudaError_t e = cudaMemcpy2DAsync(d_bufs, d_stride, h_in, h_in_stride, row, (size_t)P,
                                          cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
        int rc_ = ring_allreduce(d_bufs, d_stride, P, N, dtype, stream);
        if (rc_) return rc_;
        e = cudaMemcpy2DAsync(h_out, h_out_stride, d_bufs, d_stride, row, (size_t)P, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
        return RC_OK;
    }
    int dev;
    DeviceState *st = nullptr;
    int rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    HostPipe *hp = nullptr;
    if ((rc_ = host_pipe_streams(dev, &hp))) return rc_;
    // Events are released as soon as they are enqueued (CUDA frees them once
    // they complete); a failure part-way leaves the streams ordered.
    auto event = [](cudaEvent_t *ev) { return cudaEventCreateWithFlags(ev, cudaEventDisableTiming); };
    auto order = [&](cudaStream_t from, cudaStream_t to) -> cudaError_t {
        cudaEvent_t ev;
        cudaError_t e = event(&ev);
        if (e == cudaSuccess) e = cudaEventRecord(ev, from);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
        cudaEventDestroy(ev);
        return e;
    };
    cudaError_t e = order(s, hp->in);
    if (e == cudaSuccess) e = order(s, hp->out);
    if (e != cudaSuccess) return cuda_fail(e, "stream ordering");
    for (size_t q = 0; q < G; ++q) {
        size_t lo = c * q / G, hi = c * (q + 1) / G;
        lo -= lo % rc::kSliceGranule;
        if (q + 1 < G) hi -= hi % rc::kSliceGranule;
        const size_t n = hi - lo;
        e = copy_segment(d_bufs, d_stride, h_in, h_in_stride, P, c, lo, n, es, cudaMemcpyHostToDevice, hp->in);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
        if ((e = order(hp->in, s)) != cudaSuccess) return cuda_fail(e, "stream ordering");
        rc::RingParams p{};
        p.data = (char *)d_bufs + lo * es;
        p.data_stride = d_stride;
        p.chunk = n;
        p.chunk_stride = c;
        p.P = P;
        p.rows = 2 * (P - 1);
        p.mode = rc::MODE_ALLREDUCE;
        p.discard = 1;
        if ((rc_ = run_ring(p, dtype, s))) return rc_;
        if ((e = order(s, hp->out)) != cudaSuccess) return cuda_fail(e, "stream ordering");
        e = copy_segment(h_out, h_out_stride, d_bufs, d_stride, P, c, lo, n, es, cudaMemcpyDeviceToHost, hp->out);
        if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    }
    if ((e = order(hp->out, s)) != cudaSuccess) return cuda_fail(e, "stream ordering");
    if ((e = order(hp->in, s)) != cudaSuccess) return cuda_fail(e, "stream ordering");
    return RC_OK;
}

// Reads the header of the signal area at `ws` (device memory) after `stream`
// has completed, and clears its status word if it is set.  Returns the status
// (0 = OK) and fills *h.  Allocates nothing: the read lands in *h and the
// clear is a memset on `stream`.
static int read_and_clear_status(void *ws, cudaStream_t stream, rc::WsHeader *h, const char *what)
{
    cudaError_t e = cudaMemcpyAsync(h, ws, sizeof *h, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, what);
    if (h->status == 0) return RC_OK;
    e = cudaMemsetAsync((char *)ws + offsetof(rc::WsHeader, status), 0, sizeof(uint32_t), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return (int)h->status;
}

static void *noalloc_scratch_if_set_up(int dev);

int ring_status(void *stream)
{
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RC_OK;
    // The library's two signal areas on this device: the workspace of the
    // regular entry points and the fixed array of ring_allreduce_noalloc.
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        ws = g_dev[dev].ws;
    }
    void *na = noalloc_scratch_if_set_up(dev);
    rc::WsHeader h{}, hn{};
    const int st_ws = ws ? read_and_clear_status(ws, s, &h, "status read") : RC_OK;
    if (st_ws == RC_ERR_CUDA) return st_ws;
    const int st_na = na ? read_and_clear_status(na, s, &hn, "status read (allocation-free array)") : RC_OK;
    if (st_na == RC_ERR_CUDA) return st_na;
    if (st_ws && st_na)
        return fail(st_ws, "device wait timed out: rank %u, step %u, slice %u (and in an allocation-free call: "
                    "rank %u, step %u, slice %u)", h.err_rank, h.err_step, h.err_slice, hn.err_rank, hn.err_step,
                    hn.err_slice);
    if (st_ws)
        return fail(st_ws, "device wait timed out: rank %u, step %u, slice %u", h.err_rank, h.err_step,
                    h.err_slice);
    if (st_na)
        return fail(st_na, "device wait timed out in an allocation-free call: rank %u, step %u, slice %u",
                    hn.err_rank, hn.err_step, hn.err_slice);
    return RC_OK;
}

int ring_status_ex(void *workspace, void *stream)
{
    if (!workspace) return fail(RC_ERR_INVALID, "null workspace");
    if ((uintptr_t)workspace & 15u) return fail(RC_ERR_INVALID, "workspace must be 16-byte aligned");
    rc::WsHeader h{};
    const int st = read_and_clear_status(workspace, (cudaStream_t)stream, &h, "status read");
    if (st == RC_OK || st == RC_ERR_CUDA) return st;
    return fail(st, "device wait timed out: rank %u, step %u, slice %u", h.err_rank, h.err_step, h.err_slice);
}

// ---------------------------------------------------------------------------
// Allocation-free all-reduce.  Its scratch (workspace header + signal rows)
// is this file-scope device array instead of a cudaMalloc'd workspace.  In
// host code the name g_noalloc_scratch is only a host-side stand-in, so the
// device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint32_t g_noalloc_scratch[RC_NOALLOC_SCRATCH_BYTES / 4];

namespace {
struct NoAllocState {
    void *ptr = nullptr;     // device address of g_noalloc_scratch on this device
    uint64_t launches = 0;   // launches since the array was last cleared
};
NoAllocState g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;
} // namespace

static void *noalloc_scratch_if_set_up(int dev)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    return g_noalloc[dev].ptr;
}

int ring_allreduce_noalloc(void *bufs_base, size_t stride, int P, size_t N, int dtype, void *stream)
{
    rc::RingParams p;
    int rc_ = allreduce_params(bufs_base, stride, P, N, dtype, p);
    if (rc_ < 0) return RC_OK;
    if (rc_) return rc_;
    const size_t avail_words = (RC_NOALLOC_SCRATCH_BYTES - sizeof(rc::WsHeader)) / 4;
    const size_t words_per_slice = (size_t)P * (size_t)p.rows * (size_t)P;
    if (words_per_slice > avail_words)
        return fail(RC_ERR_INVALID, "P=%d needs %zu signal words per slice; the static scratch holds %zu (P <= 32)",
                    P, words_per_slice, avail_words);

    int dev;
    DeviceState *st = nullptr;
    rc_ = current_device(&dev, &st);
    if (rc_) return rc_;
    // The launch shape of ring_allreduce (slices, chunk segments, phase-shifted
    // rings), with the slice count then lowered until the signal rows fit in
    // the array.  Fewer slices keep every slice non-empty for the planned
    // segment count, so the segments stand.
    rc_ = plan_ring(p, dtype, st);
    if (rc_) return rc_;
    if ((size_t)p.S * words_per_slice > avail_words) p.S = (int)(avail_words / words_per_slice);

    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocState &na = g_noalloc[dev];
    cudaStream_t s = (cudaStream_t)stream;
    if (!na.ptr || na.launches >= kEpochResetAt) {
        if (!na.ptr) {
            void *ptr = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
            na.ptr = ptr;
        }
        // Signal rows and the header's epoch, done counter and status start at zero.
        cudaError_t e = cudaMemsetAsync(na.ptr, 0, RC_NOALLOC_SCRATCH_BYTES, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the static scratch");
        na.launches = 0;
    }
    p.hdr = (rc::WsHeader *)na.ptr;
    p.sig = (uint32_t *)((char *)na.ptr + sizeof(rc::WsHeader));
    p.timeout_ns = (unsigned long long)g_timeout_ms.load() * 1000000ull;
    p.skip_rank = g_skip_rank.exchange(-1);
    p.skip_step = g_skip_step.exchange(-1);
    p.trace = g_trace.load();
    p.trace_words = g_trace_words.load();
    p.debug_serial = debug_serial();
    cudaError_t e = p.pair ? rc::launch_ring_pair(p, dtype, s) : rc::launch_ring(p, dtype, rc::kRingThreads, s);
    if (e != cudaSuccess) return cuda_fail(e, "ring kernel launch");
    na.launches += (uint64_t)p.segments; // the launch advances the epoch by its segment count
    return RC_OK;
}

int ring_finalize(void)
{
    std::lock_guard<std::mutex> lock(g_mu);
    int prev = 0;
    cudaGetDevice(&prev);
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_dev[d].ws) {
            cudaSetDevice(d);
            cudaDeviceSynchronize();
            cudaFree(g_dev[d].ws);
            g_dev[d].ws = nullptr;
            g_dev[d].ws_bytes = 0;
            g_dev[d].launches = 0;
        }
        if (g_pipe[d].in) {
            cudaSetDevice(d);
            cudaStreamSynchronize(g_pipe[d].in);
            cudaStreamSynchronize(g_pipe[d].out);
            cudaStreamDestroy(g_pipe[d].in);
            cudaStreamDestroy(g_pipe[d].out);
            g_pipe[d].in = g_pipe[d].out = nullptr;
        }
    }
    cudaSetDevice(prev);
    return RC_OK;
}

} // extern "C"
