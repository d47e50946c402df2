// Work schedule shared by the persistent kernels: output tiles in groups of 8
// block rows; whole tiles dealt round-robin for all but the last one or two
// waves; the remaining tiles' K-slab iterations cut into equal contiguous
// ranges, one per CTA (stream-K). A range that starts inside a tile leaves a
// partial sum in the CTA's workspace slot, published with release flags; the
// CTA whose range holds the tile's first slab (its owner) adds the later
// CTAs' partials in CTA order, a fixed order, so results are deterministic.
// Waits only ever point to higher CTA indices, so they cannot form a cycle;
// launches with such waits must be cooperative (all CTAs resident).
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

__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until *flag != 0; false after kWaitLimitNs.
__device__ __forceinline__ bool wait_flag(const unsigned *flag)
{
    if (ld_acquire_gpu(flag) != 0) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t n = 0; n < kSpinLimit; ++n) {
        __nanosleep(64);
        if (ld_acquire_gpu(flag) != 0) return true;
        if (ptx::global_timer_ns() - t0 > ptx::kWaitLimitNs) return false;
    }
    return false;
}

// The work schedule, computed on the host (plan_schedule) and read by every
// thread of the kernel.
struct Schedule {
    int tiles_m, tiles_n;
    int64_t tiles_per_batch;   // tiles_m * tiles_n
    int nk;             // K slabs per tile
    int grid;           // CTAs launched
    int64_t tiles;      // all output tiles, batch entry after batch entry
    int64_t dp_tiles;   // whole-tile work: tiles [0, dp_tiles), round-robin
    int64_t sk_iters;   // slab iterations of the stream-K region
    int sk_ctas;        // CTAs [0, sk_ctas) share those iterations
    unsigned *flags;    // sk_ctas x (flags per CTA), zeroed before the launch
    float *partials;    // sk_ctas slots of BM x BN floats
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

// Stream-K iteration one past the last slab of stream-K tile `tile`.
__host__ __device__ __forceinline__ int64_t sk_tile_end(const Schedule &s, int64_t tile)
{
    return (tile - s.dp_tiles + 1) * s.nk;
}

// Whether CTA h, above the owner of a stream-K tile ending at iteration
// `tile_end`, still holds slabs of that tile (its range starts before the
// end). The owner's partners are g+1, g+2, ... while this holds.
__host__ __device__ __forceinline__ bool sk_holds_part(const Schedule &s, int h, int64_t tile_end)
{
    return h < s.sk_ctas && sk_start(s, h) < tile_end;
}

// For the owner g of stream-K tile `tile` (the CTA holding its first slab):
// one past the last CTA whose range holds later slabs of that tile. The
// owner adds the partial sums of CTAs g+1 .. end-1, in that order.
__host__ __device__ __forceinline__ int sk_partner_end(const Schedule &s, int g, int64_t tile)
{
    const int64_t tile_end = sk_tile_end(s, tile);
    int h = g + 1;
    while (sk_holds_part(s, h, tile_end)) ++h;
    return h;
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

// Workspace bytes of a stream-K schedule: flags (`flags_per_cta` per CTA,
// rounded to 256 bytes) then one bm x bn FP32 partial-sum slot per CTA.
size_t schedule_workspace_bytes(const Schedule &s, int flags_per_cta, int bm, int bn);

// Points the schedule's flags and partial slots into `workspace` and zeroes
// the flags on `stream`.
cudaError_t schedule_attach_workspace(Schedule &s, void *workspace, int flags_per_cta, cudaStream_t stream);

}  // namespace sgemm_gb300
