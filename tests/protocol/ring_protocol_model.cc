// ring_protocol_model.cc -- a CPU model of the ring step engine's
// synchronisation, for ThreadSanitizer (test infrastructure only).
//
// One std::thread plays one thread block (rank r, slice j, and for the
// bidirectional reduce-scatter the half h).  Chunk data are plain
// (non-atomic) uint32 words, so every cross-thread data access is a data race
// unless the signal protocol orders it: each step waits with an acquire load
// until the neighbour's signal row holds the launch's value, moves its slice,
// then stores the value to the next row of the neighbour it feeds with a
// release.  Signal values come from an epoch that the last thread of a launch
// advances by the number of segments, exactly as the kernel does, so several
// launches run back to back on one set of rows.  The schedule is the ring of
// "全归约 3：Ring——每步大小恒定" (section "走读"): reduce-scatter round s adds
// the left neighbour's chunk (r-s-2+P)%P into the own chunk of that index;
// all-gather round t copies chunk (r-1-t+P)%P from the left neighbour; the
// bidirectional variant follows "Pallas TPU Distributed Collectives 复习文档",
// section 4 (top halves travel left, bottom halves right, P-1 steps; the
// last add stores the finished half straight into its owner's output).
//
// Modes allreduce_pair and reduce_scatter_pair model the variant with two
// ranks per thread block (k_ring_pair): thread m plays ranks 2m and 2m+1,
// does rank 2m+1's step before waiting on thread m-1, hands the head of
// every slice from rank 2m to rank 2m+1 in thread-private memory (the
// kernel's shared memory), and signals only between threads.
//
// Integer adds make every order give the same sum, so the model also checks
// its results against plain sums.  Variant "early_notify" signals before the
// step's stores (a planted protocol error that ThreadSanitizer must report);
// variant "stagger" starts slice j's threads (j % 3) x 50 us late, like the
// kernel's phase-shifted slice rings.
//
// Usage: ring_protocol_model MODE P S SEGMENTS LAUNCHES N_PER_RANK [early_notify|stagger]
//   MODE: allreduce | reduce_scatter | all_gather | rs_bidir | allreduce_pair | reduce_scatter_pair |
//         rs_bidir_pair
// Exit status 0 with "ok" when every launch produced the expected result.
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

namespace {

enum Mode { ALLREDUCE, REDUCE_SCATTER, ALL_GATHER, RS_BIDIR };

struct Launch {
    Mode mode;
    bool pair;
    int P, S, segments, rows, nsteps;
    size_t chunk;                       // elements per chunk (all-gather: shard length)
    uint32_t *data;                     // P slots (all-gather: the outputs)
    size_t stride;                      // elements between slots
    const uint32_t *in;                 // all-gather inputs, P shards of `chunk`
    uint32_t *out;                      // reduce-scatter outputs, P chunks
    std::atomic<uint32_t> *sig;         // [S][P][rows][P]
    std::atomic<uint32_t> *epoch;
    std::atomic<uint32_t> *done;
    int total_threads;
    bool early_notify;
    bool stagger;
};

bool reached(uint32_t v, uint32_t want) { return (int32_t)(v - want) >= 0; }

size_t part_begin(size_t n, int i, int parts)
{
    if (i >= parts) return n;
    return n * (size_t)i / (size_t)parts;
}

void block(const Launch &L, int h, int r, int j)
{
    const int P = L.P, S = L.S;
    const bool bidir = L.mode == RS_BIDIR;
    const int left = (r - 1 + P) % P, right = (r + 1) % P;
    const int from = (bidir && h == 0) ? right : left;
    const int to = (bidir && h == 0) ? left : right;
    const uint32_t E0 = L.epoch->load(std::memory_order_relaxed);
    if (L.stagger && j % 3) std::this_thread::sleep_for(std::chrono::microseconds(50 * (j % 3)));
    std::atomic<uint32_t> *my_rows = L.sig + ((size_t)j * P + r) * L.rows * P + (size_t)h * L.nsteps * P;
    std::atomic<uint32_t> *to_rows = L.sig + ((size_t)j * P + to) * L.rows * P + (size_t)h * L.nsteps * P;
    const size_t c = L.chunk, half = c / 2;
    const size_t range_lo = bidir ? (h == 0 ? 0 : half) : 0;
    const size_t range_n = bidir ? (h == 0 ? half : c - half) : c;
    uint32_t *my = L.data + (size_t)r * L.stride;
    const uint32_t *fr = L.data + (size_t)from * L.stride;
    for (int q = 0; q < L.segments; ++q) {
        const size_t seg_lo = range_lo + part_begin(range_n, q, L.segments);
        const size_t seg_n = range_lo + part_begin(range_n, q + 1, L.segments) - seg_lo;
        const size_t lo = seg_lo + part_begin(seg_n, j, S);
        const size_t n = seg_lo + part_begin(seg_n, j + 1, S) - lo;
        const uint32_t V = E0 + 1u + (uint32_t)q;
        auto notify = [&](int row) { to_rows[(size_t)row * P + r].store(V, std::memory_order_release); };
        if (L.mode == ALL_GATHER) {
            for (size_t i = 0; i < n; ++i) my[(size_t)r * c + lo + i] = L.in[(size_t)r * c + lo + i];
            notify(0);
        }
        for (int g = 0; g < L.nsteps; ++g) {
            if (g > 0 || L.mode == ALL_GATHER) {
                std::atomic<uint32_t> &f = my_rows[(size_t)g * P + from];
                for (long spins = 0; !reached(f.load(std::memory_order_acquire), V); ++spins) {
                    if (spins > 400000000L) {
                        std::fprintf(stderr, "wait gave up: rank %d step %d slice %d\n", r, g, j);
                        std::exit(3);
                    }
                    std::this_thread::yield();
                }
            }
            const bool notify_next = g + 1 < L.nsteps;
            if (L.early_notify && notify_next) notify(g + 1);
            if (L.mode == ALL_GATHER) {
                const int k = (r - 1 - g + P) % P;
                for (size_t i = 0; i < n; ++i) my[(size_t)k * c + lo + i] = fr[(size_t)k * c + lo + i];
            } else if (bidir) {
                const int k = h == 0 ? (r + 1 + g) % P : (r - 1 - g + 2 * P) % P;
                // the last step finishes chunk k == to and stores it in that rank's output
                uint32_t *dst = g == P - 2 ? L.out + (size_t)k * c : my + (size_t)k * c;
                for (size_t i = 0; i < n; ++i) dst[lo + i] = my[(size_t)k * c + lo + i] + fr[(size_t)k * c + lo + i];
            } else if (g < P - 1) {
                const int k = (r - g - 2 + P) % P;
                uint32_t *dst = (L.mode == REDUCE_SCATTER && g == P - 2) ? L.out + (size_t)r * c : my + (size_t)k * c;
                for (size_t i = 0; i < n; ++i) dst[lo + i] = fr[(size_t)k * c + lo + i] + my[(size_t)k * c + lo + i];
            } else {
                const int k = (r - 1 - (g - (P - 1)) + P) % P;
                for (size_t i = 0; i < n; ++i) my[(size_t)k * c + lo + i] = fr[(size_t)k * c + lo + i];
            }
            if (!L.early_notify && notify_next) notify(g + 1);
        }
    }
    // the last thread of the launch publishes the new epoch
    if (L.done->fetch_add(1, std::memory_order_acq_rel) == (uint32_t)L.total_threads - 1) {
        L.done->store(0, std::memory_order_relaxed);
        L.epoch->store(E0 + (uint32_t)L.segments, std::memory_order_release);
    }
}

// Thread (h, m, j): ranks 2m and 2m+1 of ring h (h = 1 runs towards higher
// ranks; the bidirectional mode's h = 0 runs towards lower ones).  rL is fed
// by its partner in the thread, rR by the neighbouring thread.
void pair_block(const Launch &L, int h, int m, int j)
{
    const int P = L.P, S = L.S;
    const bool bidir = L.mode == RS_BIDIR, rightward = h == 1;
    const int r0 = 2 * m, r1 = 2 * m + 1;
    const int rL = rightward ? r1 : r0, rR = rightward ? r0 : r1;
    const int up = rightward ? (r0 - 1 + P) % P : (r1 + 1) % P, down = rightward ? (r1 + 1) % P : (r0 - 1 + P) % P;
    auto chunk_of = [&](int r, int s) {
        return bidir ? (rightward ? (r - 1 - s + 2 * P) % P : (r + 1 + s) % P) : (r - s - 2 + 2 * P) % P;
    };
    const uint32_t E0 = L.epoch->load(std::memory_order_relaxed);
    if (L.stagger && j % 3) std::this_thread::sleep_for(std::chrono::microseconds(50 * (j % 3)));
    const size_t row_h = bidir ? (size_t)h * L.nsteps : 0;
    std::atomic<uint32_t> *my_rows = L.sig + (((size_t)j * P + rR) * L.rows + row_h) * P;
    std::atomic<uint32_t> *to_rows = L.sig + (((size_t)j * P + down) * L.rows + row_h) * P;
    const size_t c = L.chunk, half = c / 2;
    const size_t range_lo = bidir ? (h == 0 ? 0 : half) : 0, range_n = bidir ? (h == 0 ? half : c - half) : c;
    uint32_t *s0 = L.data + (size_t)rR * L.stride, *s1 = L.data + (size_t)rL * L.stride;
    const uint32_t *sl = L.data + (size_t)up * L.stride;
    std::vector<uint32_t> hand;
    for (int q = 0; q < L.segments; ++q) {
        const size_t seg_lo = range_lo + part_begin(range_n, q, L.segments);
        const size_t seg_n = range_lo + part_begin(range_n, q + 1, L.segments) - seg_lo;
        const size_t lo = seg_lo + part_begin(seg_n, j, S);
        const size_t n = seg_lo + part_begin(seg_n, j + 1, S) - lo;
        const uint32_t V = E0 + 1u + (uint32_t)q;
        const size_t h = n / 2;   // head of the slice handed from rank r0 to r1 in private memory
        hand.assign(h, 0u);
        auto notify = [&](int row) { to_rows[(size_t)row * P + rL].store(V, std::memory_order_release); };
        for (int g = 0; g < L.nsteps; ++g) {
            const bool notify_next = g + 1 < L.nsteps;
            const bool last = g == L.nsteps - 1;
            if (L.early_notify && notify_next) notify(g + 1);
            // rank rL: needs only rank rR's previous step (this thread)
            if (g < P - 1) {
                const int k = chunk_of(rL, g);
                uint32_t *dst = (L.mode != ALLREDUCE && g == P - 2) ? L.out + (size_t)k * c : s1 + (size_t)k * c;
                for (size_t i = 0; i < n; ++i) {
                    const uint32_t a = (i < h && g >= 1) ? hand[i] : s0[(size_t)k * c + lo + i];
                    dst[lo + i] = a + s1[(size_t)k * c + lo + i];
                }
            } else {
                const int k = (rL - 1 - (g - (P - 1)) + 2 * P) % P;
                for (size_t i = 0; i < n; ++i) s1[(size_t)k * c + lo + i] = i < h ? hand[i] : s0[(size_t)k * c + lo + i];
            }
            if (!L.early_notify && notify_next) notify(g + 1);
            // rank rR: waits for the neighbouring thread (rank rR's upstream neighbour)
            if (g > 0) {
                std::atomic<uint32_t> &f = my_rows[(size_t)g * P + up];
                for (long spins = 0; !reached(f.load(std::memory_order_acquire), V); ++spins) {
                    if (spins > 400000000L) {
                        std::fprintf(stderr, "wait gave up: pair %d step %d slice %d\n", m, g, j);
                        std::exit(3);
                    }
                    std::this_thread::yield();
                }
            }
            if (g < P - 1) {
                const int k = chunk_of(rR, g);
                for (size_t i = 0; i < n; ++i) {
                    const uint32_t v = sl[(size_t)k * c + lo + i] + s0[(size_t)k * c + lo + i];
                    if (L.mode != ALLREDUCE && g == P - 2) {
                        L.out[(size_t)k * c + lo + i] = v;
                    } else if (g == P - 2) {
                        s0[(size_t)k * c + lo + i] = v;
                        if (i < h) hand[i] = v;
                    } else if (i < h) {
                        hand[i] = v;
                    } else {
                        s0[(size_t)k * c + lo + i] = v;
                    }
                }
            } else {
                const int k = (rR - 1 - (g - (P - 1)) + 2 * P) % P;
                for (size_t i = 0; i < n; ++i) {
                    const uint32_t v = sl[(size_t)k * c + lo + i];
                    s0[(size_t)k * c + lo + i] = v;
                    if (i < h && !last) hand[i] = v;
                }
            }
        }
    }
    if (L.done->fetch_add(1, std::memory_order_acq_rel) == (uint32_t)L.total_threads - 1) {
        L.done->store(0, std::memory_order_relaxed);
        L.epoch->store(E0 + (uint32_t)L.segments, std::memory_order_release);
    }
}

} // namespace

int main(int argc, char **argv)
{
    if (argc < 7) {
        std::fprintf(stderr, "usage: %s MODE P S SEGMENTS LAUNCHES N_PER_RANK [early_notify]\n", argv[0]);
        return 2;
    }
    const std::string ms = argv[1];
    const bool pair = ms == "allreduce_pair" || ms == "reduce_scatter_pair" || ms == "rs_bidir_pair";
    const Mode mode = (ms == "allreduce" || ms == "allreduce_pair") ? ALLREDUCE
                      : (ms == "reduce_scatter" || ms == "reduce_scatter_pair") ? REDUCE_SCATTER
                      : ms == "all_gather" ? ALL_GATHER : RS_BIDIR;
    const int P = std::atoi(argv[2]), S = std::atoi(argv[3]), G = std::atoi(argv[4]), launches = std::atoi(argv[5]);
    const size_t npr = (size_t)std::atoll(argv[6]);
    const bool early = argc > 7 && std::string(argv[7]) == "early_notify";
    const bool stagger = argc > 7 && std::string(argv[7]) == "stagger";
    if (P < 2 || S < 1 || G < 1 || launches < 1 || (mode != ALL_GATHER && npr % (size_t)P)) return 2;
    if (pair && (P & 1)) return 2;
    const size_t chunk = mode == ALL_GATHER ? npr : npr / (size_t)P;
    const size_t slot = mode == ALL_GATHER ? (size_t)P * npr : npr;
    const int halves = mode == RS_BIDIR ? 2 : 1;
    const int nsteps = mode == ALLREDUCE ? 2 * (P - 1) : P - 1;
    const int rows = nsteps * halves;
    std::vector<uint32_t> data((size_t)P * slot), in((size_t)P * npr), out((size_t)P * chunk);
    std::vector<std::atomic<uint32_t>> sig((size_t)S * P * rows * P);
    for (auto &w : sig) w.store(0);
    std::atomic<uint32_t> epoch{0}, done{0};
    uint64_t seed = 88172645463325252ull;
    auto rnd = [&] {
        seed ^= seed << 13;
        seed ^= seed >> 7;
        seed ^= seed << 17;
        return (uint32_t)seed;
    };
    for (int it = 0; it < launches; ++it) {
        std::vector<uint32_t> x((size_t)P * npr);
        for (auto &v : x) v = rnd();
        if (mode == ALL_GATHER) {
            in = x;
            std::fill(data.begin(), data.end(), 0u);
        } else {
            data = x;
        }
        Launch L{mode, pair, P, S, G, rows, nsteps, chunk, data.data(), slot, in.data(), out.data(), sig.data(),
                 &epoch, &done, pair ? P / 2 * S * halves : P * S * halves, early, stagger};
        std::vector<std::thread> th;
        if (pair) {
            for (int h = 0; h < halves; ++h)
                for (int m = 0; m < P / 2; ++m)
                    for (int j = 0; j < S; ++j) th.emplace_back(pair_block, std::cref(L), halves == 2 ? h : 1, m, j);
        } else {
            for (int h = 0; h < halves; ++h)
                for (int r = 0; r < P; ++r)
                    for (int j = 0; j < S; ++j) th.emplace_back(block, std::cref(L), h, r, j);
        }
        for (auto &t : th) t.join();
        // expected results: plain sums / copies
        for (size_t i = 0; i < (mode == ALL_GATHER ? 0 : npr); ++i) {
            uint32_t sum = 0;
            for (int r = 0; r < P; ++r) sum += x[(size_t)r * npr + i];
            const int k = (int)(i / chunk);
            if (mode == ALLREDUCE) {
                for (int r = 0; r < P; ++r)
                    if (data[(size_t)r * slot + i] != sum) {
                        std::printf("allreduce mismatch launch %d rank %d elem %zu\n", it, r, i);
                        return 1;
                    }
            } else if (out[(size_t)k * chunk + i % chunk] != sum) {
                std::printf("reduce-scatter mismatch launch %d chunk %d elem %zu\n", it, k, i);
                return 1;
            }
        }
        if (mode == ALL_GATHER)
            for (int r = 0; r < P; ++r)
                for (size_t i = 0; i < slot; ++i)
                    if (data[(size_t)r * slot + i] != x[i]) {
                        std::printf("all-gather mismatch launch %d rank %d elem %zu\n", it, r, i);
                        return 1;
                    }
        if (epoch.load() != (uint32_t)(G * (it + 1))) {
            std::printf("epoch %u after launch %d\n", epoch.load(), it);
            return 1;
        }
    }
    std::printf("ok\n");
    return 0;
}
