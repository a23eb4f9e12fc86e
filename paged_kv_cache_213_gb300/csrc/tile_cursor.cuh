// tile_cursor.cuh -- position in the ordered list of (KV head j, sequence b,
// 16-token tile t) work units that the split kernels walk.
//
// Units are ordered KV head j, then sequence b, then tile t, so that
// sequences holding the same physical prefix blocks (forked siblings, shared
// prompts) sit next to each other and their readers reach the shared blocks
// at about the same time (the later reads then hit L2).  pre[] is the tile
// prefix over sequences (pre[b] = tiles of sequences before b), so TB =
// pre[B] units per KV head and unit x = j * TB + pre[b] + t.
#pragma once

namespace pkv {

struct Cursor {
    int b, j, t;
};

// The unit at index x (0 <= x < Hk * pre[B]).
__device__ __forceinline__ Cursor locate(int x, const int *pre, int B) {
    const int TB = pre[B];
    const int j = x / TB;
    const int r = x - j * TB;
    int lo = 0, hi = B - 1;  // largest b with pre[b] <= r (it has tiles)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return Cursor{lo, j, r - pre[lo]};
}

// The next unit: the next tile, else the first tile of the next sequence
// that has tiles, else the next KV head.
__device__ __forceinline__ void advance(Cursor &c, const int *pre, int B) {
    if (++c.t < pre[c.b + 1] - pre[c.b]) return;
    c.t = 0;
    do {
        ++c.b;
    } while (c.b < B && pre[c.b + 1] == pre[c.b]);
    if (c.b < B) return;
    ++c.j;
    c.b = 0;
    while (c.b < B && pre[c.b + 1] == pre[c.b]) ++c.b;
}

}  // namespace pkv
