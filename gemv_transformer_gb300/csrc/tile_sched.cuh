// tile_sched.cuh -- what the tensor-core GEMV kernels share besides the arithmetic:
// the copies that feed their stages, the consumer warps' named barrier, the routing
// of a MoE launch's slots, and the schedule of 16-row tiles over the CTAs.
//
// Routing follows hanzo-ml 0.11.13 src/wgpu_backend.rs, moe_matvec_gpu: slot s is
// (token s / topk, expert ids[s]) and its output row is y[s] = W[ids[s]] . x[s / topk].
// A CTA takes the slots in windows of kMaxSlots, sorts a window by (expert, slot) and
// cuts it into segments of one expert each; a slot whose id lies outside
// [0, n_experts) is reported (kStBadExpert) and left out.
#pragma once

#include <cuda.h>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {

constexpr int kMaxSlots = 256;  // slots per routing window

// One box of a 3-D tensor map (weight bank [matrix][row][k]) into shared memory,
// completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y,
                                            int z, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// Global -> shared bulk copy completing on `bar`, default L2 policy (X is read by
// every CTA); 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_g2s_nohint(void *dst, const void *src, uint32_t bytes,
                                                uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Named barrier 1 over the CW consumer warps of a CTA (the producer warp is not in it).
template <int CW>
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory");
}

// The same barrier, returning whether any consumer thread passed `v` true.  Every
// consumer gets the same answer, so a decision taken on it (leave, or go on to the
// next barrier) is taken by all of them together -- unlike a read of a flag after
// the barrier, which a warp outside it (the producer) may set in between.
template <int CW>
__device__ __forceinline__ bool consumers_sync_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(CW * 32)
        : "memory");
    return r != 0;
}

// Shared-memory tables of one routing window.
struct RouteSmem {
    unsigned long long *key;  // [kMaxSlots], 16-byte aligned: 64-bit keys, or 32-bit keys then their ranks
    int *sorted;              // [kMaxSlots]: the global slot index of each rank
    int *seg;                 // [kMaxSlots + 1]: segment starts, then the valid slots' end
    int *act;                 // [kMaxSlots]: the expert of each segment
    int *nact;                // the number of segments
    int *wcnt;                // [kMaxSlots / 32]: per-warp counts of segment starts
};

// Routes slots [base, base + Sl) (1 <= Sl <= kMaxSlots).  Every thread of the block
// calls it, with blockDim.x >= kMaxSlots; the tables are complete after the caller's
// next __syncthreads.
__device__ __forceinline__ void route_window(const StreamArgs &a, int base, int Sl,
                                             const RouteSmem &rs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool k32_ok = a.n_experts < (1 << 24) - 1;
    uint32_t *k32 = reinterpret_cast<uint32_t *>(rs.key);
    if (k32_ok) {
        // 32-bit keys expert << 8 | slot (a bad id as expert 0xFFFFFF), padded to a
        // whole number of 16-byte quads with keys that rank below none; each key's
        // rank is counted by up to four threads over slices of the quads.
        int *s_rank = reinterpret_cast<int *>(k32 + kMaxSlots);
        for (int i = threadIdx.x; i < Sl; i += blockDim.x) {
            const int e = a.ids[base + i];
            const bool okid = e >= 0 && e < a.n_experts;
            if (!okid && blockIdx.x == 0) record_status(a.status, kStBadExpert);
            k32[i] = ((okid ? (uint32_t)e : 0xFFFFFFu) << 8) | (uint32_t)i;
            s_rank[i] = 0;
        }
        const int nq = (Sl + 3) / 4;
        if ((int)threadIdx.x < 4 * nq - Sl) k32[Sl + threadIdx.x] = 0xFFFFFFFFu;
        __syncthreads();
        const int parts = max(1, min(4, (int)blockDim.x / Sl));
        const int qper = (nq + parts - 1) / parts;
        for (int idx = threadIdx.x; idx < Sl * parts; idx += blockDim.x) {
            const int part = idx / Sl, i = idx - part * Sl;
            const uint32_t ki = k32[i];
            int r = 0;
            const int q1 = min(nq, (part + 1) * qper);
            for (int q = part * qper; q < q1; ++q) {
                const uint4 kk = reinterpret_cast<const uint4 *>(k32)[q];
                r += (int)(kk.x < ki) + (int)(kk.y < ki) + (int)(kk.z < ki) + (int)(kk.w < ki);
            }
            atomicAdd(&s_rank[i], r);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < Sl; i += blockDim.x) rs.sorted[s_rank[i]] = base + i;
    } else {
        const unsigned long long big = 1ull << 62;
        for (int i = threadIdx.x; i < Sl; i += blockDim.x) {
            const int e = a.ids[base + i];
            const bool okid = e >= 0 && e < a.n_experts;
            if (!okid && blockIdx.x == 0) record_status(a.status, kStBadExpert);
            rs.key[i] = okid ? ((unsigned long long)e << 16) | (unsigned)i : big | (unsigned)i;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < Sl; i += blockDim.x) {
            const unsigned long long ki = rs.key[i];
            int r = 0;
            for (int i2 = 0; i2 < Sl; ++i2) r += rs.key[i2] < ki;
            rs.sorted[r] = base + i;  // the slot's global index
        }
    }
    __syncthreads();
    // The expert of the r-th sorted slot, or -1 for a bad id.
    auto sorted_expert = [&](int r) -> int {
        const int i = rs.sorted[r] - base;
        if (k32_ok) {
            const uint32_t e = k32[i] >> 8;
            return e == 0xFFFFFFu ? -1 : (int)e;
        }
        const unsigned long long kr = rs.key[i];
        return (kr >> 62) ? -1 : (int)(kr >> 16);
    };
    // Segments of the sorted slots, one thread per position: position r starts one
    // when its expert differs from r - 1's, and the starts are numbered by a count
    // over the warps' ballots.
    const int r = threadIdx.x;
    int e = -1;
    bool start = false, last = false;
    if (r < Sl) {
        e = sorted_expert(r);
        start = e >= 0 && (r == 0 || sorted_expert(r - 1) != e);
        last = e >= 0 && (r == Sl - 1 || sorted_expert(r + 1) < 0);
    }
    const unsigned bm = __ballot_sync(0xFFFFFFFFu, start);
    if (lane == 0 && warp < kMaxSlots / 32) rs.wcnt[warp] = __popc(bm);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < (Sl + 31) / 32; ++w) {
        const int c = rs.wcnt[w];
        before += w < warp ? c : 0;
        total += c;
    }
    if (start) {
        const int idx = before + __popc(bm & ((1u << lane) - 1u));
        rs.seg[idx] = r;
        rs.act[idx] = e;
    }
    if (last) {  // the valid slots end here (bad ids sort last)
        rs.seg[total] = r + 1;
        *rs.nact = total;
    }
    if (r == 0 && e < 0) {  // no valid slot in the window
        rs.seg[0] = 0;
        *rs.nact = 0;
    }
}

// ------------------------------------------------------------ job schedule --
//
// Work units are 16-row tiles; GEMV: tiles 0..ceil(m/16) of the one matrix; MoE:
// tiles of the active experts (expert a owns units [a*tpe, (a+1)*tpe)).  A CTA
// processes its units in row groups of at most T tiles that never straddle an
// expert, each group once per pass of the tokens that fit in one: the GEMV's CTAs
// take contiguous ranges (split_units, Walk), the MoE's the groups dealt out by
// cost (DealWalk).

struct Sched {
    int n_act;          // MoE: active experts; GEMV: 1
    int tpe;            // tiles per expert (GEMV: per matrix)
    long long u0, u1;   // this CTA's unit range
};

// This CTA's contiguous share of the sc.n_act * sc.tpe units (the GEMV's split).
__device__ __forceinline__ void split_units(Sched &sc) {
    const long long units = (long long)sc.n_act * sc.tpe;
    if (units * gridDim.x < (1ll << 32)) {  // the usual case: 32-bit divisions
        const uint32_t uu = (uint32_t)units;
        sc.u0 = uu * blockIdx.x / gridDim.x;
        sc.u1 = uu * (blockIdx.x + 1) / gridDim.x;
    } else {
        sc.u0 = units * blockIdx.x / gridDim.x;
        sc.u1 = units * (blockIdx.x + 1) / gridDim.x;
    }
}

// MoE: the active experts (segment indices) by ascending slot count, ties by
// index: order[i] is the i-th.  Every thread of the block calls it; the table is
// complete after the caller's next __syncthreads.
__device__ __forceinline__ void order_by_slots(const int *seg, int n_act, int *order) {
    for (int a = threadIdx.x; a < n_act; a += blockDim.x) {
        const int na = seg[a + 1] - seg[a];
        int r = 0;
        for (int b = 0; b < n_act; ++b) {
            const int nb = seg[b + 1] - seg[b];
            r += (nb < na) || (nb == na && b < a);
        }
        order[r] = a;
    }
}

// A walk over the CTA's unit range by row groups.  The position (slot ai among
// the active experts, tile tl within it) is advanced by addition: one division
// when the walk starts, none per group or per chunk.
struct Walk {
    long long u, u1;  // next unit, end of the range
    int ai, tl, tpe;
    __device__ __forceinline__ explicit Walk(const Sched &sc) : u(sc.u0), u1(sc.u1), tpe(sc.tpe) {
        ai = u < (1ll << 32) ? (int)((uint32_t)u / (uint32_t)tpe) : (int)(u / tpe);
        tl = (int)(u - (long long)ai * tpe);
    }
    __device__ __forceinline__ bool more() const { return u < u1; }
    // Tiles in the next group: at most T, never past the expert or the range.
    template <int T>
    __device__ __forceinline__ int group() const {
        long long e = T < tpe - tl ? T : tpe - tl;
        if (e > u1 - u) e = u1 - u;
        return (int)e;
    }
    __device__ __forceinline__ void advance(int nt) {
        u += nt;
        tl += nt;
        if (tl == tpe) {
            tl = 0;
            ++ai;
        }
    }
};

// MoE: a CTA's row groups dealt out by cost.  Each active expert's tiles form gpe
// groups of T (the last one shorter when T does not divide tpe), and a group's
// cost grows with its expert's slot count (more or wider passes).  The groups are
// ranked by that count (`order`, from order_by_slots) and CTA b takes ranks b,
// 2 grid - 1 - b, 2 grid + b, ...: the rounds alternate direction, so a CTA that
// took one of the cheapest groups of a round takes one of the dearest of the next.
// (With fewer groups than CTAs some CTAs stay idle: the launcher picks T with that
// in view.)  Same interface as Walk: `ai` the active expert, `tl` the group's
// first tile.
template <int T>
struct DealWalk {
    const int *order;
    int tpe, gpe, G, b, grid, r, rank, ai, tl;
    __device__ __forceinline__ DealWalk(const Sched &sc, const int *order_)
        : order(order_), tpe(sc.tpe), gpe((sc.tpe + T - 1) / T), G(sc.n_act * gpe),
          b((int)blockIdx.x), grid((int)gridDim.x), r(0) {
        locate();
    }
    __device__ __forceinline__ void locate() {
        rank = r * grid + ((r & 1) ? grid - 1 - b : b);
        if (rank < G) {
            const int sp = rank / gpe;
            ai = order[sp];
            tl = (rank - sp * gpe) * T;
        }
    }
    __device__ __forceinline__ bool more() const { return rank < G; }
    template <int TT>
    __device__ __forceinline__ int group() const { return T < tpe - tl ? T : tpe - tl; }
    __device__ __forceinline__ void advance(int) {
        ++r;
        locate();
    }
};


}  // namespace wq
