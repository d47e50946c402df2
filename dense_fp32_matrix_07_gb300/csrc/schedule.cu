// Host side of the shared work schedule (see schedule.cuh).
#include "schedule.cuh"

namespace sgemm_gb300 {

namespace {
size_t round_up_bytes(size_t x, size_t a) { return (x + a - 1) / a * a; }
size_t counter_bytes(const Schedule &s, int counters_per_tile)
{
    return round_up_bytes((size_t)(s.tiles - s.dp_tiles) * counters_per_tile * sizeof(unsigned), 256);
}
}  // namespace

Schedule plan_schedule(int64_t M, int64_t N, int64_t K, int bm, int bn, int bk, int64_t slots, int policy,
                       bool with_sk, int64_t batch)
{
    Schedule s{};
    s.tiles_m = (int)((M + bm - 1) / bm);
    s.tiles_n = (int)((N + bn - 1) / bn);
    s.nk = (int)((K + bk - 1) / bk);
    s.k_last = (int)(K - (int64_t)(s.nk - 1) * bk);
    s.tiles_per_batch = (int64_t)s.tiles_m * s.tiles_n;
    s.tiles = s.tiles_per_batch * (batch > 0 ? batch : 1);
    s.dp_tiles = s.tiles;
    s.sk_iters = 0;
    s.sk_ctas = 0;
    s.grid = (int)(s.tiles < slots ? s.tiles : slots);
    if (with_sk && policy == kSchedTailSplit) {
        // Leftover tiles of the last, partial wave are each cut into `parts`
        // equal K ranges, one per CTA: the ranges start together at aligned
        // K offsets, so the tail runs as `parts` lockstep fronts.
        const int64_t full_rounds = s.tiles / slots;
        const int64_t rem = s.tiles - full_rounds * slots;
        const int64_t parts = rem > 0 ? slots / rem : 0;
        if (parts >= 2 && s.nk >= 2 * parts) {
            s.dp_tiles = full_rounds * slots;
            s.sk_iters = rem * s.nk;
            s.sk_ctas = (int)(rem * parts);
            s.grid = (int)(s.dp_tiles > 0 ? slots : s.sk_ctas);
        }
        return s;
    }
    bool sk = false;
    if (with_sk && policy == kSchedStreamK) {
        sk = true;
    } else if (with_sk && policy == kSchedAuto) {
        const int64_t rounds = (s.tiles + slots - 1) / slots;
        // With at least one full wave ahead of it, a partial last wave is
        // worth evening out as soon as it idles 0.5 % of the slots (128 x 256
        // tiles, same-box A/B against whole tiles: 3072^3 0.867 vs 0.903 ms,
        // 8192^3 16.05 vs 16.66 ms, 12288^3 54.08 vs 55.29 ms; 16384^3, 99.8 %
        // full, stays whole). A single partial wave, where every tile would
        // be split, only below 90 % (at 1536^3 on 128 x 128 tiles, 144 tiles
        // on 152 SMs, whole tiles measured 123.1 us against 126.1 us).
        const double fill = (double)s.tiles / (double)(rounds * slots);
        sk = s.nk >= 8 && (rounds >= 2 ? fill < 0.995 : fill < 0.90);
    }
    if (!sk) return s;
    // Stream-K covers the leftover tiles of the last, partial wave, and also
    // the last full wave when the leftover fills less than a third of the
    // slots (a short region would otherwise cut each tile into many parts).
    // Leftover alone against leftover + one wave, same-box A/B: 2048^3
    // 268.9 against 270.4 us, 3072^3 852.0 against 854.1 us, 4096^3 1975.2
    // against 1975.9 us; fewer tiles run split, so fewer operand slabs are
    // read at scattered K offsets.
    const int64_t full_rounds = s.tiles / slots;
    const int64_t leftover = s.tiles - full_rounds * slots;
    const int64_t dp_rounds = (policy == kSchedStreamK || full_rounds < 1) ? 0
                              : (3 * leftover >= slots ? full_rounds : full_rounds - 1);
    s.dp_tiles = dp_rounds * slots;
    s.sk_iters = (s.tiles - s.dp_tiles) * s.nk;
    const int64_t min_iters = policy == kSchedStreamK ? 1 : 4;
    int64_t ctas = s.sk_iters / min_iters;
    if (ctas > slots) ctas = slots;
    if (ctas < 1) ctas = 1;
    s.sk_ctas = (int)ctas;
    s.grid = (int)(s.dp_tiles > 0 ? slots : ctas);
    return s;
}

size_t schedule_workspace_bytes(const Schedule &s, int counters_per_tile, int bm, int bn)
{
    if (s.sk_ctas == 0) return 0;
    return counter_bytes(s, counters_per_tile) + 2 * (size_t)s.sk_ctas * bm * bn * sizeof(float);
}

size_t schedule_counter_bytes(const Schedule &s, int counters_per_tile)
{
    return s.sk_ctas == 0 ? 0 : counter_bytes(s, counters_per_tile);
}

cudaError_t schedule_attach_workspace(Schedule &s, void *workspace, int counters_per_tile, bool zero,
                                      cudaStream_t stream)
{
    const size_t cb = counter_bytes(s, counters_per_tile);
    s.counters = static_cast<unsigned *>(workspace);
    s.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + cb);
    return zero ? cudaMemsetAsync(s.counters, 0, cb, stream) : cudaSuccess;
}

}  // namespace sgemm_gb300
