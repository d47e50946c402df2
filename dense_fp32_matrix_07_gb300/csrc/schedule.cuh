// Work schedule shared by the persistent kernels: output tiles in groups of 8
// block rows; whole tiles dealt round-robin for all but the last one or two
// waves; the remaining tiles' K-slab iterations cut into equal contiguous
// ranges, one per CTA (stream-K). A tile whose slabs fall in several CTAs'
// ranges is reduced by whichever of them finishes its part last: each part
// that is not last writes its partial sum to a slot of its own and counts
// itself in the tile's arrival counter; the part that completes the count
// adds every part in CTA order (a fixed order, so results are
// deterministic) and stores the tile. No CTA ever waits for another, so no
// launch needs all its CTAs resident at once.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace sgemm_gb300 {

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Adds 1 with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned atomic_inc_acq_rel_gpu(unsigned *p)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
}

// The work schedule, computed on the host (plan_schedule) and read by every
// thread of the kernel.
struct Schedule {
    int tiles_m, tiles_n;
    int64_t tiles_per_batch;   // tiles_m * tiles_n
    int nk;             // K slabs per tile
    int k_last;         // k of the last slab that hold data (1 .. bk)
    int grid;           // CTAs launched
    int64_t tiles;      // all output tiles, batch entry after batch entry
    int64_t dp_tiles;   // whole-tile work: tiles [0, dp_tiles), round-robin
    int64_t sk_iters;   // slab iterations of the stream-K region
    int sk_ctas;        // CTAs [0, sk_ctas) share those iterations
    unsigned *counters; // arrival counters: (tiles - dp_tiles) x (counters per tile), zeroed before the launch
    float *partials;    // 2 x sk_ctas slots of BM x BN floats (sk_slot)
};

// One unit of work: slabs [kb0, kb1) of output tile `tile`.
struct Item {
    int64_t tile;
    int kb0, kb1;
};

struct Cursor {
    int64_t dp_next;        // next whole tile of this CTA
    int64_t sk_pos, sk_end; // this CTA's stream-K iteration range
};

__host__ __device__ __forceinline__ int64_t sk_start(const Schedule &s, int g)
{
    return s.sk_iters * g / s.sk_ctas;
}

// The CTAs whose ranges hold slabs of stream-K tile `tile` are
// sk_first_cta .. sk_last_cta. CTA g's range starts at floor(S g / C)
// (S = sk_iters, C = sk_ctas), so the CTA holding iteration x is the largest
// g with floor(S g / C) <= x, i.e. ceil((x + 1) C / S) - 1. Every range is
// non-empty (plan_schedule keeps sk_ctas <= sk_iters).
__host__ __device__ __forceinline__ int sk_cta_of_iter(const Schedule &s, int64_t x)
{
    return (int)(((x + 1) * s.sk_ctas + s.sk_iters - 1) / s.sk_iters - 1);
}

__host__ __device__ __forceinline__ int sk_first_cta(const Schedule &s, int64_t tile)
{
    return sk_cta_of_iter(s, (tile - s.dp_tiles) * s.nk);
}

__host__ __device__ __forceinline__ int sk_last_cta(const Schedule &s, int64_t tile)
{
    return sk_cta_of_iter(s, (tile - s.dp_tiles + 1) * s.nk - 1);
}

// Partial-sum slot of CTA g's part of a split tile. A CTA holds at most two
// such parts: the first item of its range, which may start inside a tile
// (kb0 > 0), and the last, which may end inside one (it then starts at the
// tile's first slab). They take slots 2g and 2g + 1, so no slot is written
// twice in one launch. The part of sk_first_cta is the one starting at slab 0.
__host__ __device__ __forceinline__ int64_t sk_slot(int g, int kb0)
{
    return 2 * (int64_t)g + (kb0 == 0 ? 1 : 0);
}

__host__ __device__ __forceinline__ int64_t sk_part_slot(int h, int first)
{
    return sk_slot(h, h == first ? 0 : 1);
}

__host__ __device__ __forceinline__ Cursor cursor_init(const Schedule &s, int g)
{
    Cursor c;
    c.dp_next = g;
    if (g < s.sk_ctas) {
        c.sk_pos = sk_start(s, g);
        c.sk_end = sk_start(s, g + 1);
    } else {
        c.sk_pos = c.sk_end = 0;
    }
    return c;
}

__host__ __device__ __forceinline__ bool next_item(const Schedule &s, Cursor &c, Item &it)
{
    if (c.dp_next < s.dp_tiles) {
        it.tile = c.dp_next;
        it.kb0 = 0;
        it.kb1 = s.nk;
        c.dp_next += s.grid;
        return true;
    }
    if (c.sk_pos < c.sk_end) {
        const int64_t rel = c.sk_pos / s.nk;
        it.tile = s.dp_tiles + rel;
        it.kb0 = (int)(c.sk_pos - rel * s.nk);
        const int64_t left = c.sk_end - c.sk_pos;
        it.kb1 = (int)(left < s.nk - it.kb0 ? it.kb0 + left : s.nk);
        c.sk_pos += it.kb1 - it.kb0;
        return true;
    }
    return false;
}

// Output tile of linear index t: groups of 8 block rows, column-major inside
// a group, so the CTAs running at the same time touch few A and B panels.
__host__ __device__ __forceinline__ void tile_coords(int64_t t, int tiles_m, int tiles_n, int &tm, int &tn)
{
    constexpr int GR = 8;
    const int64_t per_group = (int64_t)GR * tiles_n;
    const int64_t group = t / per_group;
    const int first_m = (int)(group * GR);
    const int rows = tiles_m - first_m < GR ? tiles_m - first_m : GR;
    const int64_t local = t - group * per_group;
    tm = first_m + (int)(local % rows);
    tn = (int)(local / rows);
}

// Batch entry and tile of linear tile index t (batch entries one after the
// other, the grouped order within each).
__host__ __device__ __forceinline__ void tile_coords_b(const Schedule &s, int64_t t, int &b, int &tm, int &tn)
{
    const int64_t bb = t / s.tiles_per_batch;
    b = (int)bb;
    tile_coords(t - bb * s.tiles_per_batch, s.tiles_m, s.tiles_n, tm, tn);
}

// ------------------------------- host side -------------------------------

// Plans the schedule of an M x N x K product in bm x bn tiles with bk-deep
// slabs on `slots` resident CTAs. Policy (SchedPolicy): whole tiles; forced
// stream-K over every tile, split down to one slab per CTA (for tests);
// automatic: stream-K only when a tile spans at least 8 slabs and whole
// tiles would leave slots idle: more than 0.5 % of them when at least one
// full wave precedes the last, more than 10 % when all tiles fit in one
// partial wave; it keeps at least 4 slabs per CTA; or tail split: whole tiles for every full wave, then each leftover
// tile cut into floor(slots / leftover) >= 2 equal K parts. `with_sk` false
// always gives whole tiles. Pointers are left null.
Schedule plan_schedule(int64_t M, int64_t N, int64_t K, int bm, int bn, int bk, int64_t slots, int policy,
                       bool with_sk, int64_t batch = 1);

// Workspace bytes of a stream-K schedule: the arrival counters
// (`counters_per_tile` per stream-K tile, rounded up to 256 bytes), then two
// bm x bn FP32 partial-sum slots per CTA of the stream-K region.
size_t schedule_workspace_bytes(const Schedule &s, int counters_per_tile, int bm, int bn);

// Bytes of the arrival counters at the start of that workspace (0 without a
// stream-K region).
size_t schedule_counter_bytes(const Schedule &s, int counters_per_tile);

// Points the schedule's counters and partial slots into `workspace` and, if
// `zero`, zeroes the counters on `stream` (else the caller has).
cudaError_t schedule_attach_workspace(Schedule &s, void *workspace, int counters_per_tile, bool zero,
                                      cudaStream_t stream);

}  // namespace sgemm_gb300
