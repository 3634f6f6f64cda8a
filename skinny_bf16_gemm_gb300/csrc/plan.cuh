// Work split of the decode GEMM (shared by the host planner and the kernel).
//
// The weight W[N, K] is cut into tiles of 128 rows (one MMA M extent) and each
// tile's K range into blocks of 64 (one 128-byte swizzle row of BF16). The
// tiles * kblocks weight blocks, in tile-major order, are cut into G contiguous
// ranges of (almost) equal length ("stream-K"), one per persistent CTA: every CTA
// streams the same number of weight bytes whatever N and K are, so no SM idles
// in a partial last wave. A tile whose K range spans several ranges is finished
// by the CTA whose range holds the tile's first K blocks, which adds the others'
// FP32 partial sums in K order.
//
// Ranges are numbered in K order (range r precedes range r + 1) and dealt to
// CTAs in reverse block order (range r to block G - 1 - r). A tile's finisher
// holds its lowest range, so it has the highest block index of the tile's
// contributors, and every CTA it waits for has a lower block index: blocks are
// dispatched in index order, so those are already running (or done) whatever
// else occupies the GPU, and the waits never depend on all G CTAs being
// resident at once.
#pragma once

#include <cstdint>

namespace skinny {

constexpr int kBlockN = 128;       // weight rows per tile = MMA M
constexpr int kBlockK = 64;        // K per pipeline stage: 128 bytes of BF16
constexpr int kMaxM = 64;          // rows of x (MMA N is 16, 32 or 64)
constexpr int kSlotFloats = kMaxM * kBlockN;  // one FP32 partial tile [m][row] (device scratch)

struct GemmGeometry {
    int M, N, K;
    int tiles;        // ceil(N / 128)
    int kblocks;      // ceil(K / 64)
    long long blocks; // tiles * kblocks
    int ctas;         // G
};

__host__ __device__ inline GemmGeometry make_geometry(int M, int N, int K, int num_sms) {
    GemmGeometry g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.tiles = (N + kBlockN - 1) / kBlockN;
    g.kblocks = (K + kBlockK - 1) / kBlockK;
    g.blocks = static_cast<long long>(g.tiles) * g.kblocks;
    g.ctas = static_cast<int>(g.blocks < num_sms ? g.blocks : num_sms);
    return g;
}

// CTAs to launch on a device with num_sms SMs. When the tiles alone nearly fill
// the GPU (at least 90 % of the SMs), each CTA takes one whole tile: no tile is
// shared, so there is no split-K fix-up, and the few idle SMs cost less than the
// fix-ups would. Otherwise one CTA per SM with the stream-K split.
__host__ __device__ inline int choose_ctas(int N, int num_sms) {
    const int tiles = (N + kBlockN - 1) / kBlockN;
    if (tiles <= num_sms && tiles * 10 >= num_sms * 9) return tiles;
    return num_sms;
}

// Ring depth. A deep ring (one CTA per SM) keeps the most weight bytes in flight
// and wins on long streams; a shallow one lets the next kernel's CTA share the
// SM under programmatic dependent launch, which wins when each CTA streams
// little (the next kernel's set-up and first weights then matter more). Measured
// on GB300 the two cross near 1 MiB of weights per CTA, and near 1.5 MiB for up
// to 16 rows of x, whose shallow ring is deepest (6 stages): between 1 and 1.5
// MiB it is 0.3-0.45 us faster there, level for 32 rows, 3.5-5 us slower for 64.
// More than 32 rows never take it: their shallow ring could hold only 4 stages,
// and the deep ring was 0.6-1 us faster even at N = 2048-4096.
constexpr long long kShallowRingMaxBytes = 1ll << 20;
constexpr long long kShallowRingMaxBytes16 = 3ll << 19;

__host__ __device__ inline bool use_shallow_ring(const GemmGeometry &g, bool pdl) {
    const long long per_cta = g.blocks * (kBlockN * kBlockK * 2) / g.ctas;
    return pdl && g.M <= 32 &&
           per_cta < (g.M <= 16 ? kShallowRingMaxBytes16 : kShallowRingMaxBytes);
}

// Range of the CTA with block index b, and the block index of the CTA that
// streams range r (the map is its own inverse).
__host__ __device__ inline int range_of_block(const GemmGeometry &g, int b) { return g.ctas - 1 - b; }

// In the functions below c is a range index, not a block index.

// First weight block of range c (c = ctas gives the end of the last range).
__host__ __device__ inline long long cta_begin(const GemmGeometry &g, int c) {
    return (g.blocks * c) / g.ctas;
}

// The range holding weight block i: the largest c with cta_begin(c) <= i.
__host__ __device__ inline int block_owner(const GemmGeometry &g, long long i) {
    return static_cast<int>(((i + 1) * g.ctas - 1) / g.blocks);
}

// Scratch slot of range c's partial sum for tile t: two per range, one for the
// tile it starts in and one for the tile it ends in.
__host__ __device__ inline int partial_slot(const GemmGeometry &g, int c, int t) {
    return 2 * c + (t == static_cast<int>(cta_begin(g, c) / g.kblocks) ? 0 : 1);
}

// Piece q of range c: tile t, blocks [kb0, kb1) of it.
struct Piece {
    int tile, kb0, kb1;
};

__host__ __device__ inline int cta_piece_count(const GemmGeometry &g, int c) {
    long long b0 = cta_begin(g, c), b1 = cta_begin(g, c + 1);
    if (b1 <= b0) return 0;
    return static_cast<int>((b1 - 1) / g.kblocks - b0 / g.kblocks + 1);
}

__host__ __device__ inline Piece cta_piece(const GemmGeometry &g, int c, int q) {
    long long b0 = cta_begin(g, c), b1 = cta_begin(g, c + 1);
    int t = static_cast<int>(b0 / g.kblocks) + q;
    long long t0 = static_cast<long long>(t) * g.kblocks;
    Piece p;
    p.tile = t;
    p.kb0 = static_cast<int>((b0 > t0 ? b0 : t0) - t0);
    p.kb1 = static_cast<int>((b1 < t0 + g.kblocks ? b1 : t0 + g.kblocks) - t0);
    return p;
}

// A walk over consecutive weight blocks in tile-major order without divisions
// (64-bit integer division is a long software sequence on the GPU).
struct BlockCursor {
    int t, kb;  // tile, K block within it
    __host__ __device__ void next(int kblocks) {
        if (++kb == kblocks) {
            kb = 0;
            ++t;
        }
    }
};

// Ranges contributing to tile t, in K order: [first, last].
__host__ __device__ inline void tile_contributors(const GemmGeometry &g, int t, int &first,
                                                  int &last) {
    long long t0 = static_cast<long long>(t) * g.kblocks;
    first = block_owner(g, t0);
    last = block_owner(g, t0 + g.kblocks - 1);
}

}  // namespace skinny
