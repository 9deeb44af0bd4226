// Stream-K schedule of the tensor-core projections, shared by the kernels
// that produce split-tile partials and the kernels that consume them.
//
// A unit is one (batch chunk, 128-row tile, run of KU 64-wide k tiles); units
// are numbered tile-major (u = tile * KT + j, tile = chunk * MT + mt, where KT
// here counts units per row tile).  CTA c of
// G takes units [c*U/G, (c+1)*U/G).  The part of a tile's KT units that one
// CTA covers is a segment; segment `slot` of a tile is the one done by CTA
// (first CTA of the tile) + slot.  A tile's partial sums live at
// part[((tile * max_seg + slot) * 64 + b) * 128 + r] (b = sequence in the
// chunk, r = row in the tile) and the result is the sum over its segments in
// slot order.  The CTA that produces a tile's last segment also writes the
// tile's segment count to nseg[tile], so consumers need one load, not a
// search.  Unit counts stay below 2^31 / G (checked on the host), so the
// schedule uses 32-bit arithmetic.
#pragma once

namespace dn {

struct SchedView {
    int U, G, KT, MT, max_seg;
};

__host__ __device__ inline int sched_unit_start(int c, const SchedView &s) {
    return (int)(((unsigned)c * (unsigned)s.U) / (unsigned)s.G);
}

// the CTA whose unit range holds unit u
__host__ __device__ inline int sched_cta_of_unit(int u, const SchedView &s) {
    int lo = 0, hi = s.G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sched_unit_start(mid, s) <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// number of segments (partials) of a tile
__host__ __device__ inline int sched_nseg(int tile, const SchedView &s) {
    return sched_cta_of_unit(tile * s.KT + s.KT - 1, s) - sched_cta_of_unit(tile * s.KT, s) + 1;
}

}  // namespace dn
