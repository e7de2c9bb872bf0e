// Kernel-map build for submanifold convolution: for every active voxel, the input
// index of each of its 27 neighbours (-1 when absent).
//
// The submanifold variant (outputs only at active sites; "pixal3d_mrp_mlx
// CLAUDE.md", "Measured facts": stride 1 / no padding dispatches to SubMConv3d)
// needs exactly this table; the pages' "spatial cache" (README scope table) is what
// lets one table serve several convolutions on one voxel set.
//
// Pipeline (one stream; a synchronous build waits once, at the end, for the status
// word). Sort key of a voxel: (b << 3*bits) | Morton(z, y, x), bits >= 2 per axis. The
// low 6 bits of a Morton code are the voxel's place inside its aligned 4x4x4 block and
// the bits above name the block, so the Morton order is the order of the occupied
// blocks by key, each block's voxels by place.
//   1. insert  : validate each coordinate; find or claim its block's slot in an
//                open-addressing hash table (splitmix64 of the block key, bounded linear
//                probing, atomicCAS) and OR its bit into the slot's 64-bit occupancy
//                mask
//   2. compact : the occupied slots (block key, slot index)
//   3. sort    : LSD radix sort of the block keys only (single-pass passes with
//                decoupled look-back; passes whose digit is constant are skipped)
//   4. starts  : exclusive scan of the sorted blocks' popcounts: each block's first
//                position, stored in its slot; fewer positions than voxels (all of them
//                valid and inserted) is a duplicate coordinate
//   5. scatter : a voxel's position = its block's first position + the rank of its
//                bit; (sort key, input row) stored there: the Morton order
//   6. probe   : warps take 32 consecutive positions; per run of one block they look
//                up the (at most 27) neighbour blocks the run's voxels reach, then each
//                lane resolves its voxel's 27 neighbours by a bit test and a popcount
//                (position = neighbour block's first position + rank), whose input row
//                is the answer; rows are staged in shared memory and written out whole.
// The radix sort of all N voxels' keys (pack, histograms, passes, block runs, table)
// is kept for the downsample's own sort, for builds whose table would exceed 2^31
// slots, and to name the first repeated row when a build finds a duplicate.
// The blocks of a shell hold ~10 voxels each, so the table is about a tenth of a
// per-voxel table and stays in L2.
// Hash of a block key: the splitmix64 finaliser (Steele, Lea and Flood, 2014).
//
// The structure ops that share the radix sort live here too (their section is below the
// probe): SparseDownsample(2), which numbers the parents of the sorted voxels and pools
// their features; SparseUpsample(2), its cache-paired inverse; SparseSpatial2Channel(2)
// and its inverse, the sparse pixel-(un)shuffle on the same subdivision.
#include "common.cuh"

namespace subm3d {
namespace {

constexpr unsigned long long kEmptyKey = ~0ull;
constexpr int kSortThreads = 256;
constexpr int kSortItems = 8;   // 2048-key tiles: ~80 registers, three blocks per SM
constexpr int kSortTile = kSortThreads * kSortItems;   // keys per sort block
constexpr int kMaxPasses = 8;
constexpr int kMaxProbe = 4096;
constexpr int kHistParts = 16;   // partial digit histograms (spreads the count kernel's atomics)
// shared memory of a sort pass over tiles of `tile` keys
constexpr int scatter_smem(int tile) { return tile * 12 + (kSortThreads / 32) * 257 * 4 + 2 * 256 * 4; }
// The block-key sort runs on a twelfth as many keys: quarter-size tiles give it four
// times as many blocks in flight (its passes are latency-bound at that size).
constexpr int kBlockSortItems = 2;
constexpr int kSmallTileRatio = kSortItems / kBlockSortItems;

enum : int {
  kFlagCoord = 1, kFlagDup = 2, kFlagFull = 4, kFlagInternal = 8, kFlagOrder = 16,
  kFlagGrow = 32,   // hashed front end: the first table was too small, rebuilt at full size
};

struct KmapStatus {
  int flags;
  int pad;
  long long bad_row;
  int plan[kMaxPasses + 1];   // plan[p]: bit1 = pass active, bit0 = source buffer; plan[8] = final buffer
  int pad2;
  int plan2[kMaxPasses + 1];  // the same for the grouping sort of the tile plan
  int pad3;
  unsigned long long nblocks;    // occupied 4x4x4 blocks
  unsigned long long cap;        // hash capacity in use (a power of two)
  unsigned long long kmin, kmax; // smallest and largest sort key
  unsigned long long npos;       // positions of the block-grouped order the probe walks
  unsigned int scan_ctr;         // next tile of the block-start scan
  unsigned int pad4;
};

struct __align__(32) Slot {
  unsigned long long key;    // block key, kEmptyKey when free
  unsigned long long mask;   // bit (Morton order of the voxel inside the block) per active voxel
  unsigned long long start;  // first sorted position of the block's voxels
  unsigned long long pad;    // (one 32-byte load brings the whole slot)
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Radix-sort scratch for ntile 2048-key tiles: tile counters (256 bytes), digit starts of
// every pass, and the published per-tile digit counts.
__host__ __device__ inline size_t sort_scratch_bytes(int64_t ntile) {
  return 256 + sizeof(uint32_t) * kMaxPasses * 256 +
         sizeof(unsigned long long) * size_t(ntile) * 256;
}

struct Layout {
  // bv1: the second value buffer of the hashed front end's block sort (ix1 holds each
  // voxel's slot meanwhile)
  size_t status, hist, mk0, mk1, ix0, ix1, bv1, cnt, table;
  // tile plan only: grouping-sort keys and values (ping-pong), its histograms, and the
  // neighbour table in sorted (Morton) order
  size_t k2a, k2b, v2a, v2b, hist2, nbr_sorted;

  size_t total;
  int64_t nblk;
};

Layout make_layout(int64_t N, int64_t cap, bool grouped = false) {
  Layout L;
  L.nblk = (N + kSortTile - 1) / kSortTile;
  const size_t hist_bytes = sizeof(uint32_t) * kHistParts * kMaxPasses * 256;
  size_t o = 0;
  L.status = o; o = align256(o + sizeof(KmapStatus));
  L.hist = o;   o = align256(o + hist_bytes);
  L.mk0 = o;    o = align256(o + sizeof(uint64_t) * N);
  L.mk1 = o;    o = align256(o + sizeof(uint64_t) * N);
  L.ix0 = o;    o = align256(o + sizeof(int32_t) * N);
  L.ix1 = o;    o = align256(o + sizeof(int32_t) * N);
  L.bv1 = o;    o = align256(o + sizeof(int32_t) * N);
  L.cnt = o;    o = align256(o + sort_scratch_bytes(L.nblk * kSmallTileRatio));
  L.table = o;  o = align256(o + sizeof(Slot) * cap);
  L.k2a = L.k2b = L.v2a = L.v2b = L.hist2 = L.nbr_sorted = 0;
  if (grouped) {
    L.k2a = o;      o = align256(o + sizeof(uint64_t) * N);
    L.k2b = o;      o = align256(o + sizeof(uint64_t) * N);
    L.v2a = o;      o = align256(o + sizeof(int32_t) * N);
    L.v2b = o;      o = align256(o + sizeof(int32_t) * N);
    L.hist2 = o;    o = align256(o + hist_bytes);
    L.nbr_sorted = o; o = align256(o + sizeof(int32_t) * 27 * N);
  }
  L.total = o;
  return L;
}

// Bit t of v (v < 2^21) to bit 3t, and back: the usual shift-and-mask bit interleave,
// each step moving half of the remaining bit groups apart (or together).
__host__ __device__ __forceinline__ unsigned long long spread3(uint32_t v) {
  unsigned long long x = v & 0x1fffffu;
  x = (x | (x << 32)) & 0x1f00000000ffffull;
  x = (x | (x << 16)) & 0x1f0000ff0000ffull;
  x = (x | (x << 8)) & 0x100f00f00f00f00full;
  x = (x | (x << 4)) & 0x10c30c30c30c30c3ull;
  x = (x | (x << 2)) & 0x1249249249249249ull;
  return x;
}
__host__ __device__ __forceinline__ uint32_t compact3(unsigned long long x) {
  x &= 0x1249249249249249ull;
  x = (x | (x >> 2)) & 0x10c30c30c30c30c3ull;
  x = (x | (x >> 4)) & 0x100f00f00f00f00full;
  x = (x | (x >> 8)) & 0x1f0000ff0000ffull;
  x = (x | (x >> 16)) & 0x1f00000000ffffull;
  x = (x | (x >> 32)) & 0x1fffffull;
  return static_cast<uint32_t>(x);
}
// Morton code of (z, y, x): bit t of x -> 3t, of y -> 3t+1, of z -> 3t+2.
__device__ __forceinline__ unsigned long long morton3(uint32_t z, uint32_t y, uint32_t x) {
  return spread3(x) | (spread3(y) << 1) | (spread3(z) << 2);
}


__device__ __forceinline__ unsigned long long mix64(unsigned long long v) {
  v = (v ^ (v >> 30)) * 0xbf58476d1ce4e5b9ull;
  v = (v ^ (v >> 27)) * 0x94d049bb133111ebull;
  return v ^ (v >> 31);
}

// 1. ------------------------------------------------------------------------------
__global__ void kmap_init(KmapStatus* st, uint32_t* hist, uint32_t* hist2) {
  const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  if (tid == 0) {
    st->flags = 0;
    st->pad = 0;
    st->bad_row = 0x7FFFFFFFFFFFFFFFll;
    for (int p = 0; p <= kMaxPasses; ++p) st->plan[p] = st->plan2[p] = 0;
    st->pad2 = st->pad3 = 0;
    st->nblocks = 0;
    st->cap = 0;
    st->kmin = ~0ull;
    st->kmax = 0;
    st->npos = 0;
    st->scan_ctr = 0;
    st->pad4 = 0;
  }
  for (int64_t i = tid; i < kHistParts * kMaxPasses * 256; i += stride) {
    hist[i] = 0;
    if (hist2) hist2[i] = 0;
  }
}

// 2. ------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) kmap_pack(const int4* __restrict__ coords, int64_t N,
                                                 int res, int bits,
                                                 unsigned long long* __restrict__ mk,
                                                 int32_t* __restrict__ ix, KmapStatus* st) {
  unsigned long long lo = ~0ull, hi = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < N; i += stride) {
    int4 c = coords[i];   // (b, z, y, x)
    const bool ok = static_cast<unsigned>(c.x) <= SUBM3D_MAX_BATCH &&
                    static_cast<unsigned>(c.y) < static_cast<unsigned>(res) &&
                    static_cast<unsigned>(c.z) < static_cast<unsigned>(res) &&
                    static_cast<unsigned>(c.w) < static_cast<unsigned>(res);
    if (!ok) {
      atomicOr(&st->flags, kFlagCoord);
      atomicMin(&st->bad_row, static_cast<long long>(i));
      c = make_int4(0, 0, 0, 0);
    }
    const unsigned long long m =
        (static_cast<unsigned long long>(c.x) << (3 * bits)) | morton3(c.y, c.z, c.w);
    mk[i] = m;
    ix[i] = static_cast<int32_t>(i);
    lo = m < lo ? m : lo;
    hi = m > hi ? m : hi;
  }
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    const unsigned long long h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    lo = l2 < lo ? l2 : lo;
    hi = h2 > hi ? h2 : hi;
  }
  // one pair of atomics per block (same-address atomics from every warp serialise)
  __shared__ unsigned long long wlo[8], whi[8];
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    wlo[warp] = lo;
    whi[warp] = hi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) {
      lo = wlo[w] < lo ? wlo[w] : lo;
      hi = whi[w] > hi ? whi[w] : hi;
    }
    atomicMin(&st->kmin, lo);
    atomicMax(&st->kmax, hi);
  }
}

// 3. ------------------------------------------------------------------------------
// N >= 0: the sort is of all N voxels, and the order the probe walks holds every one.
__global__ void kmap_plan(int npass, int64_t N, KmapStatus* st) {
  if (N >= 0) st->npos = static_cast<unsigned long long>(N);
  const unsigned long long diff = st->kmax ^ st->kmin;
  int buf = 0;
  for (int p = 0; p < kMaxPasses; ++p) {
    const bool active = p < npass && (diff >> (8 * p)) != 0;
    st->plan[p] = active ? (2 | buf) : 0;
    if (active) buf ^= 1;
  }
  st->plan[kMaxPasses] = buf;
}

// The grouping sort of the tile plan runs every one of its npass passes.
__global__ void kmap_plan2(int npass, KmapStatus* st) {
  for (int p = 0; p < kMaxPasses; ++p) st->plan2[p] = p < npass ? (2 | (p & 1)) : 0;
  st->plan2[kMaxPasses] = npass & 1;
}

// 4. Single-pass LSD radix sort passes (decoupled look-back, after Merrill and Garland's
// single-pass prefix scan, 2016, as used for radix sorting by Adinets and Merrill's
// Onesweep, 2022). Before the passes, one read of the keys gives every pass's digit
// histogram, hence each digit's global start. A pass is then one kernel: a block takes
// the next 2048-key tile (tile numbers handed out in start order by an atomic counter,
// so a tile only ever waits for tiles whose blocks are already running), ranks its keys
// per digit in shared memory, publishes its per-digit counts, and, per digit, walks back
// over the earlier tiles' published values (a tile's own count, or the count of keys
// in that tile and all before it) until it has the number of keys of that digit before
// its own; it publishes that inclusive count in turn and writes each digit's run of its
// keys contiguously. Every wait is bounded; a wait that runs out flags the build as
// failed (internal error) and goes on with what it has.
constexpr int kWarpsPerSort = kSortThreads / 32;
// A published status word: (pass + 1) << 34 | kind << 32 | count. One array serves every
// pass of a sort (it is cleared before the sort's first pass); the pass tag tells a
// word of the current pass from one an earlier pass left.
constexpr unsigned long long kTileAggregate = 1ull << 32;   // count of this tile only
constexpr unsigned long long kTileInclusive = 2ull << 32;   // count through this tile

struct SortScratch {          // in the workspace: counters | digit starts | tile status
  uint32_t* counter;          // [kMaxPasses] next tile number of each pass
  uint32_t* gofs;             // [kMaxPasses][256] first sorted position of each digit
  unsigned long long* status; // [ntile][256] published per-digit counts (pass-tagged)
};
inline SortScratch sort_scratch(char* base, int64_t ntile) {
  SortScratch S;
  S.counter = reinterpret_cast<uint32_t*>(base);
  S.gofs = reinterpret_cast<uint32_t*>(base + 256);
  S.status = reinterpret_cast<unsigned long long*>(base + 256 + sizeof(uint32_t) * kMaxPasses * 256);
  (void)ntile;
  return S;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// 4a. Digit histograms of every pass from one read of the keys (kHistParts partial
// histograms [part][pass][digit] spread the atomics); also clears the passes' tile
// counters and published status words.
__global__ void __launch_bounds__(256) kmap_hist(const unsigned long long* __restrict__ keys,
                                                 int64_t N, const unsigned long long* count,
                                                 int npass, const int* plans,
                                                 uint32_t* __restrict__ hist, SortScratch S,
                                                 int64_t ntile, int tile_keys) {
  if (count && *count < static_cast<unsigned long long>(N)) N = static_cast<int64_t>(*count);
  __shared__ uint32_t sh[kMaxPasses][256];
  for (int i = threadIdx.x; i < kMaxPasses * 256; i += 256) sh[i >> 8][i & 255] = 0;
  const int64_t gtid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  if (gtid < kMaxPasses) S.counter[gtid] = 0;
  // the status words of the tiles that hold keys (the passes' other blocks return at once)
  const int64_t used = (N + tile_keys - 1) / tile_keys;
  const int64_t nstat = (used < ntile ? used : ntile) * 256;
  for (int64_t i = gtid; i < nstat; i += stride) S.status[i] = 0;
  unsigned active = 0;   // passes that run (a constant digit's pass is skipped)
  for (int p = 0; p < npass; ++p)
    if (plans[p] & 2) active |= 1u << p;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  // whole warps take part in every round (warp-aggregated counts: keys of nearby rows
  // share their high digits)
  for (int64_t w0 = gtid - lane; w0 < N; w0 += stride) {
    const int64_t i = w0 + lane;
    const bool valid = i < N;
    const unsigned long long k = valid ? keys[i] : 0ull;
    for (int p = 0; p < npass; ++p) {
      if (!((active >> p) & 1u)) continue;
      const uint32_t d = valid ? static_cast<uint32_t>((k >> (8 * p)) & 255u) : 256u;
      const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
      if (__all_sync(0xffffffffu, d == d0)) {   // one digit for the whole warp (common)
        if (lane == 0 && d0 < 256u) atomicAdd(&sh[p][d0], 32u);
      } else if (valid) {                      // a few lanes per digit: plain atomics
        atomicAdd(&sh[p][d], 1u);
      }
    }
  }
  __syncthreads();
  for (int p = 0; p < npass; ++p) {
    const uint32_t v = sh[p][threadIdx.x];
    if (v) atomicAdd(&hist[((blockIdx.x % kHistParts) * kMaxPasses + p) * 256 + threadIdx.x], v);
  }
}

// Exclusive prefix sum of one value per thread over a 256-thread block; returns the
// thread's prefix and leaves the block total in *total. `tmp` holds 8 words.
__device__ __forceinline__ uint32_t block_exclusive_scan256(uint32_t x, uint32_t* tmp,
                                                            uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = x;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  uint32_t wpre = 0, all = 0;
  for (int w = 0; w < 8; ++w) {
    const uint32_t t = tmp[w];
    if (w < warp) wpre += t;
    all += t;
  }
  __syncthreads();
  *total = all;
  return wpre + incl - x;
}

// 4b. One block of 256 threads: each pass's digit starts (exclusive scan of its histogram).
__global__ void __launch_bounds__(256) kmap_digit_starts(const uint32_t* __restrict__ hist,
                                                         int npass, SortScratch S) {
  __shared__ uint32_t tmp[8];
  for (int p = 0; p < npass; ++p) {
    uint32_t c = 0;
    for (int q = 0; q < kHistParts; ++q) c += hist[(q * kMaxPasses + p) * 256 + threadIdx.x];
    uint32_t total;
    S.gofs[p * 256 + threadIdx.x] = block_exclusive_scan256(c, tmp, &total);
  }
}

// 4c. One pass: rank a tile, look back for each digit's count before it, scatter.
template <int ITEMS>
__global__ void __launch_bounds__(kSortThreads) kmap_onesweep(
    unsigned long long* mk0, unsigned long long* mk1, int32_t* ix0, int32_t* ix1, int64_t N,
    const unsigned long long* count, int pass, int64_t ntile, const int* plans, SortScratch S,
    KmapStatus* st) {
  const int plan = plans[pass];
  if (!(plan & 2)) return;
  // a count on the device: N is then only the bound the grid was sized for
  if (count && *count < static_cast<unsigned long long>(N)) N = static_cast<int64_t>(*count);
  (void)ntile;
  const unsigned long long* src = (plan & 1) ? mk1 : mk0;
  unsigned long long* dst = (plan & 1) ? mk0 : mk1;
  const int32_t* isrc = (plan & 1) ? ix1 : ix0;
  int32_t* idst = (plan & 1) ? ix0 : ix1;
  constexpr int kTile = kSortThreads * ITEMS;           // keys per tile
  constexpr int kPerWarp = kTile / kWarpsPerSort;
  constexpr int kRounds = kPerWarp / 32;                // = ITEMS
  extern __shared__ __align__(16) unsigned char sort_sm[];
  unsigned long long* skey = reinterpret_cast<unsigned long long*>(sort_sm);
  int32_t* srow = reinterpret_cast<int32_t*>(sort_sm + kTile * 8);
  uint32_t* wcnt = reinterpret_cast<uint32_t*>(sort_sm + kTile * 12);   // [kWarps][257]
  uint32_t* loff = wcnt + kWarpsPerSort * 257;                                // [256]
  uint32_t* gbase = loff + 256;                                               // [256]
  __shared__ uint32_t tmp[8];
  __shared__ uint32_t s_tile;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // A block takes tiles until none are left (the grid is what fits on the GPU at once;
  // every tile is taken by a running block, so a look-back only ever waits for tiles
  // that running blocks hold).
  for (;;) {
    if (threadIdx.x == 0) s_tile = atomicAdd(&S.counter[pass], 1u);
    for (int i = threadIdx.x; i < kWarpsPerSort * 257; i += kSortThreads) wcnt[i] = 0;
    __syncthreads();
    const int64_t tile = s_tile;
    // past the last tile (tiles are handed out in order, so no tile that holds keys waits
    // for one past the end)
    if (tile * kTile >= N) return;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int64_t tile0 = tile * kTile;
    const int64_t base = tile0 + warp * kPerWarp;
    unsigned long long key[kRounds];
    int32_t row[kRounds];
    uint32_t rank[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int64_t e = base + r * 32 + lane;
      const bool valid = e < N;
      key[r] = valid ? src[e] : 0ull;
      row[r] = valid ? isrc[e] : 0;
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const bool valid = base + r * 32 + lane < N;
      const uint32_t d = valid ? static_cast<uint32_t>((key[r] >> (8 * pass)) & 255u) : 256u;
      const unsigned peers = __match_any_sync(0xffffffffu, d);
      const uint32_t before = __popc(peers & lt_mask);
      const uint32_t prior = wcnt[warp * 257 + d];
      __syncwarp();
      if (before == 0) wcnt[warp * 257 + d] = prior + __popc(peers);
      __syncwarp();
      rank[r] = prior + before;
    }
    __syncthreads();
    const int d = threadIdx.x;   // this thread's digit from here on
    uint32_t run = 0;            // keys of digit d in this tile
    for (int w = 0; w < kWarpsPerSort; ++w) {
      const uint32_t c = wcnt[w * 257 + d];
      wcnt[w * 257 + d] = run;
      run += c;
    }
    {
      uint32_t total;
      loff[d] = block_exclusive_scan256(run, tmp, &total);
    }
    // publish this tile's count, then look back for the count before it
    const unsigned long long tag = static_cast<unsigned long long>(pass + 1) << 34;
    unsigned long long* my = S.status + tile * 256 + d;
    uint32_t before_tile = 0;
    if (tile == 0) {
      st_relaxed_u64(my, tag | kTileInclusive | run);
    } else {
      st_relaxed_u64(my, tag | kTileAggregate | run);
      // eight earlier tiles' words are read at once; the walk goes on from the first one
      // not yet published (waiting for it, bounded) until an inclusive count ends it
      int64_t t = tile - 1;
      const unsigned long long t0 = global_timer_ns();
      bool late = false;
      for (uint32_t it = 0; t >= 0; ++it) {
        unsigned long long v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[q] = t - q >= 0 ? ld_relaxed_u64(S.status + (t - q) * 256 + d)
                            : (tag | kTileInclusive);   // before tile 0: nothing
        int used = 0;
        bool done = false;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (done || used < q) continue;   // stopped at an unpublished word
          const unsigned long long flag = (v[q] >> 34) == static_cast<unsigned long long>(pass + 1)
                                              ? (v[q] & (3ull << 32)) : 0ull;
          if (flag == 0) continue;          // not published yet (or an earlier pass's word)
          before_tile += static_cast<uint32_t>(v[q]);
          ++used;
          if (flag == kTileInclusive) done = true;
        }
        if (done) break;
        t -= used;
        if (used < 8 && (it & 63u) == 63u && global_timer_ns() - t0 > kWaitLimitNs) {
          late = true;
          break;
        }
      }
      if (late) atomicOr(&st->flags, kFlagInternal);
      st_relaxed_u64(my, tag | kTileInclusive | (before_tile + run));
    }
    gbase[d] = S.gofs[pass * 256 + d] + before_tile;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int64_t e = base + r * 32 + lane;
      if (e < N) {
        const uint32_t dd = static_cast<uint32_t>((key[r] >> (8 * pass)) & 255u);
        const uint32_t local = loff[dd] + wcnt[warp * 257 + dd] + rank[r];
        skey[local] = key[r];
        srow[local] = row[r];
      }
    }
    __syncthreads();
    const int nvalid = static_cast<int>((N - tile0) < kTile ? (N - tile0) : kTile);
    for (int i = threadIdx.x; i < nvalid; i += kSortThreads) {
      const unsigned long long k = skey[i];
      const uint32_t dd = static_cast<uint32_t>((k >> (8 * pass)) & 255u);
      const int64_t pos = int64_t(gbase[dd]) + (i - static_cast<int>(loff[dd]));
      if (pos >= 0 && pos < N) {
        dst[pos] = k;
        idst[pos] = srow[i];
      } else {
        atomicOr(&st->flags, kFlagInternal);
      }
    }
    __syncthreads();   // the tile's shared arrays are free for the next one
  }
}

// 5. ------------------------------------------------------------------------------
// Over the sorted order: duplicates (adjacent equal codes; the stable sort puts the
// later input row second), block runs counted, the order written if asked for.
__global__ void __launch_bounds__(256) kmap_blocks_count(
    const unsigned long long* __restrict__ mk0, const unsigned long long* __restrict__ mk1,
    const int32_t* __restrict__ ix0, const int32_t* __restrict__ ix1, int64_t N,
    int32_t* __restrict__ order, KmapStatus* st) {
  const bool second = st->plan[kMaxPasses] & 1;
  const unsigned long long* mk = second ? mk1 : mk0;
  const int32_t* ix = second ? ix1 : ix0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  unsigned long long starts = 0;
  for (int64_t s = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; s < N; s += stride) {
    const unsigned long long m = mk[s];
    const int32_t row = ix[s];
    if (static_cast<uint64_t>(row) >= static_cast<uint64_t>(N)) atomicOr(&st->flags, kFlagInternal);
    if (order) order[s] = row;
    if (s == 0) {
      ++starts;
    } else {
      const unsigned long long prev = mk[s - 1];
      if ((prev >> 6) != (m >> 6)) ++starts;
      if (prev == m) {
        atomicOr(&st->flags, kFlagDup);
        atomicMin(&st->bad_row, static_cast<long long>(row));
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) starts += __shfl_xor_sync(0xffffffffu, starts, o);
  // one atomic per block (same-address atomics from every warp serialise)
  __shared__ unsigned long long wsum[8];
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = starts;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long total = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += wsum[w];
    if (total) atomicAdd(&st->nblocks, total);
  }
}

// 6. ------------------------------------------------------------------------------
// Capacity in use: the caller's, or the smallest power of two >= 2 x blocks (>= 64,
// <= the workspace's). Clears exactly that many slots.
__global__ void kmap_table_init(Slot* table, int64_t cap_fixed, int64_t cap_max, KmapStatus* st) {
  unsigned long long cap = static_cast<unsigned long long>(cap_fixed);
  if (cap == 0) {
    cap = 64;
    while (cap < 2 * st->nblocks && cap < static_cast<unsigned long long>(cap_max)) cap <<= 1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) st->cap = cap;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
       i < static_cast<int64_t>(cap); i += stride) {
    Slot s;
    s.key = kEmptyKey;
    s.mask = 0;
    s.start = 0;
    s.pad = 0;
    table[i] = s;
  }
}

// 7. ------------------------------------------------------------------------------
// A warp takes 32 consecutive sorted positions. Each lane's bit (its code's low 6
// bits) is OR-ed into the first lane of its block's run by a segmented scan over
// shuffles (runs are contiguous); the run's first lane inserts the block with its key
// (the sort key without its low 6 bits: the batch and the Morton code of the block's
// coordinates) and first sorted position. A run that goes on past the warp's last lane
// is finished from memory by its first lane (a run holds at most 64 distinct codes;
// longer runs are duplicates, reported in step 5).
__global__ void __launch_bounds__(256) kmap_blocks_insert(
    const int4* __restrict__ coords, const unsigned long long* __restrict__ mk0,
    const unsigned long long* __restrict__ mk1, const int32_t* __restrict__ ix0,
    const int32_t* __restrict__ ix1, int64_t N, Slot* table,
    KmapStatus* st) {
  const bool second = st->plan[kMaxPasses] & 1;
  const unsigned long long* mk = second ? mk1 : mk0;
  (void)ix0;
  (void)ix1;
  const unsigned long long cap = st->cap;
  const unsigned long long cmask = cap - 1;
  const int max_probe = cap < kMaxProbe ? static_cast<int>(cap) : kMaxProbe;
  const int lane = threadIdx.x & 31;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t w0 = blockIdx.x * int64_t(blockDim.x) + threadIdx.x - lane; w0 < N; w0 += stride) {
    const int64_t s = w0 + lane;
    const bool live = s < N;
    const unsigned long long m = live ? mk[s] : ~0ull;
    const unsigned long long blk = m >> 6;
    unsigned long long prev = __shfl_up_sync(0xffffffffu, blk, 1);
    if (lane == 0) prev = (s > 0 && live) ? (mk[s - 1] >> 6) : ~0ull;
    const bool start = live && (s == 0 || prev != blk);
    unsigned long long acc = live ? (1ull << (m & 63u)) : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {   // OR of the lanes [lane, lane + 2 off) of the run
      const unsigned long long o = __shfl_down_sync(0xffffffffu, acc, off);
      const unsigned long long ob = __shfl_down_sync(0xffffffffu, blk, off);
      if (lane + off < 32 && ob == blk) acc |= o;
    }
    const unsigned long long last_blk = __shfl_sync(0xffffffffu, blk, 31);
    // the run that reaches lane 31 may go on: its bits among the next 64 positions (a run
    // without duplicates holds at most 64 voxels), loaded by the whole warp at once
    unsigned long long tail = 0;
    if (w0 + 31 < N) {   // lane 31 holds a voxel (warp-uniform)
      unsigned long long t_or = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t j = w0 + 32 + 32 * h + lane;
        const unsigned long long mj = j < N ? mk[j] : ~0ull;
        // only the stretch that continues the run without a break counts
        const unsigned brk = __ballot_sync(0xffffffffu, (mj >> 6) != last_blk);
        const unsigned keep = brk ? ((1u << (__ffs(brk) - 1)) - 1u) : 0xffffffffu;
        if ((keep >> lane) & 1u) t_or |= 1ull << (mj & 63u);
        for (int o = 16; o > 0; o >>= 1) t_or |= __shfl_xor_sync(0xffffffffu, t_or, o);
        if (brk) break;
      }
      tail = t_or;
    }
    if (start) {
      unsigned long long mask = acc;
      if (blk == last_blk) mask |= tail;   // the run reaches lane 31: add what follows
      const unsigned long long key = blk;
      unsigned long long h = mix64(key) & cmask;
      int probe = 0;
      for (; probe < max_probe; ++probe) {
        const unsigned long long prevk = atomicCAS(&table[h].key, kEmptyKey, key);
        if (prevk == kEmptyKey) {
          table[h].mask = mask;
          table[h].start = static_cast<unsigned long long>(s);
          break;
        }
        if (prevk == key) {   // two runs of one block: only possible for rejected coordinates
          atomicOr(&st->flags, kFlagInternal);
          break;
        }
        h = (h + 1) & cmask;
      }
      if (probe == max_probe) atomicOr(&st->flags, kFlagFull);
    }
  }
}

// 7h. -----------------------------------------------------------------------------
// Hashed front end. The probe needs an order of the voxels in which every occupied
// 4x4x4 block is one contiguous run, with each block's slot giving its occupancy mask
// and first position. The Morton order is such an order, and it is also the order of
// the occupied blocks by their keys, each block's voxels by their place in it (the low
// 6 bits of the code). So instead of sorting the N voxels' codes, the blocks are found
// first and only their keys are sorted (about a tenth as many on surfaces):
//   insert : each voxel finds or claims its block's slot and ORs its bit into the
//            slot's mask;
//   compact: the occupied slots' keys and indices, with the smallest and largest key;
//   sort   : the LSD radix sort of (block key, slot) (count read on the device);
//   starts : an exclusive scan of the sorted blocks' popcounts (per-tile sums, a scan
//            of those, then each block's first position into its slot); fewer
//            positions than voxels is a duplicate coordinate;
//   scatter: each voxel's position is its block's first position plus the rank of its
//            bit in the mask; its sort key and input row (and the order, if asked for)
//            go there.
// The result is the Morton order the radix sort of all voxels gives (positions of
// distinct codes; ties exist only with duplicates, which fail the build). The table is
// first sized for N/4 blocks (shells hold about ten voxels per block); a block needing
// more than kGrowProbe probes there marks the build, and the table is cleared and
// filled again at the workspace's full capacity (>= 2N slots).
constexpr int kGrowProbe = 32;

// Status word for a hashed build, the digit histograms, and the first table cleared.
__global__ void kmap_h_init(Slot* table, unsigned long long cap, uint32_t* hist,
                            uint32_t* hist2, KmapStatus* st) {
  const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  if (tid == 0) {
    st->flags = 0;
    st->pad = 0;
    st->bad_row = 0x7FFFFFFFFFFFFFFFll;
    for (int p = 0; p <= kMaxPasses; ++p) st->plan[p] = st->plan2[p] = 0;
    st->pad2 = st->pad3 = 0;
    st->nblocks = 0;
    st->cap = cap;
    st->kmin = ~0ull;
    st->kmax = 0;
    st->npos = 0;
    st->scan_ctr = 0;
    st->pad4 = 0;
  }
  for (int64_t i = tid; i < kHistParts * kMaxPasses * 256; i += stride) {
    hist[i] = 0;
    if (hist2) hist2[i] = 0;
  }
  const Slot empty{kEmptyKey, 0ull, 0ull, 0ull};
  for (int64_t i = tid; i < static_cast<int64_t>(cap); i += stride) table[i] = empty;
}

// The full-capacity table, only when the first one was too small.
__global__ void kmap_h_grow(Slot* table, unsigned long long cap, KmapStatus* st) {
  if (!(st->flags & kFlagGrow)) return;
  const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (tid == 0) st->cap = cap;
  const Slot empty{kEmptyKey, 0ull, 0ull, 0ull};
  for (int64_t i = tid; i < static_cast<int64_t>(cap); i += int64_t(gridDim.x) * blockDim.x)
    table[i] = empty;
}

// kSkip: the voxel takes no position (a coordinate out of range, or a block that did not
// fit).
constexpr uint32_t kSkip = 0xFFFFFFFFu;

__device__ __forceinline__ bool coord_ok(int4 c, int res) {   // (b, z, y, x)
  return static_cast<unsigned>(c.x) <= SUBM3D_MAX_BATCH &&
         static_cast<unsigned>(c.y) < static_cast<unsigned>(res) &&
         static_cast<unsigned>(c.z) < static_cast<unsigned>(res) &&
         static_cast<unsigned>(c.w) < static_cast<unsigned>(res);
}
__device__ __forceinline__ unsigned long long sort_key(int4 c, int bits) {
  return (static_cast<unsigned long long>(c.x) << (3 * bits)) | morton3(c.y, c.z, c.w);
}

// refill: the second launch, which runs only when the first table was too small.
// can_grow: a block needing more than kGrowProbe probes marks the build for the
// full-size table instead of failing. Each voxel looks its block up on its own (a read
// first, atomicCAS only on an empty slot), then ORs its bit into the mask as a reduction
// that returns nothing (duplicates show up later as fewer mask bits than voxels).
// (Grouping a warp's lanes by block with match/reduce intrinsics, ORing the bits of
// consecutive lanes in one block with shuffles before a single atomic per run, reading
// back the old mask, or four voxels per thread -- fewer warps then fit -- each measured
// slower; two voxels per thread at 32 registers keep every warp resident.)
__global__ void __launch_bounds__(256, 8) kmap_h_insert(const int4* __restrict__ coords,
                                                        int64_t N, int res, int bits, Slot* table,
                                                        uint32_t* __restrict__ slot_of,
                                                        bool refill, bool can_grow,
                                                        KmapStatus* st) {
  if (refill && !(st->flags & kFlagGrow)) return;
  const unsigned long long cap = st->cap;
  const unsigned long long cmask = cap - 1;
  const int max_probe = cap < kMaxProbe ? static_cast<int>(cap) : kMaxProbe;
  const int limit = can_grow ? (kGrowProbe < max_probe ? kGrowProbe : max_probe) : max_probe;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  // two voxels per round (i and i + stride): their coordinate loads and first slot reads
  // are in flight together, at a register count that keeps every warp resident
  for (int64_t i0 = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i0 < N; i0 += 2 * stride) {
    int4 c[2];
    c[0] = coords[i0];
    c[1] = i0 + stride < N ? coords[i0 + stride] : make_int4(-1, 0, 0, 0);
    unsigned long long key[2], hh[2], k0[2];
    bool ok[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t i = i0 + u * stride;
      ok[u] = i < N && coord_ok(c[u], res);
      if (i < N && !ok[u]) {
        atomicOr(&st->flags, kFlagCoord);
        atomicMin(&st->bad_row, static_cast<long long>(i));
      }
      key[u] = sort_key(c[u], bits);
      hh[u] = mix64(key[u] >> 6) & cmask;
      k0[u] = ok[u] ? __ldcg(&table[hh[u]].key) : 0ull;
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= N) break;
      uint32_t sidx = kSkip;
      if (ok[u]) {
        const unsigned long long blk = key[u] >> 6;
        unsigned long long h = hh[u], k = k0[u];
        long long found = -1;
        for (int probe = 0; probe < limit; ++probe) {
          if (probe > 0) k = __ldcg(&table[h].key);
          if (k == kEmptyKey) k = atomicCAS(&table[h].key, kEmptyKey, blk);
          if (k == kEmptyKey || k == blk) {
            found = static_cast<long long>(h);
            break;
          }
          h = (h + 1) & cmask;
        }
        if (found < 0) {
          atomicOr(&st->flags, can_grow ? kFlagGrow : kFlagFull);
        } else {
          atomicOr(&table[found].mask, 1ull << (key[u] & 63u));
          sidx = static_cast<uint32_t>(found);
        }
      }
      slot_of[i] = sidx;
    }
  }
}

// The occupied slots (key, index), 256 slots per block and round, and the smallest and
// largest key (for the sort's constant digits).
__global__ void __launch_bounds__(256) kmap_h_compact(const Slot* __restrict__ table,
                                                      unsigned long long* __restrict__ bkey,
                                                      int32_t* __restrict__ bslot,
                                                      KmapStatus* st) {
  __shared__ uint32_t tmp[8];
  __shared__ unsigned long long s_base, wlo[8], whi[8];
  const unsigned long long cap = st->cap;
  unsigned long long lo = ~0ull, hi = 0;
  for (unsigned long long b0 = blockIdx.x * 256ull; b0 < cap; b0 += gridDim.x * 256ull) {
    const unsigned long long i = b0 + threadIdx.x;
    const unsigned long long k = i < cap ? __ldcg(&table[i].key) : kEmptyKey;
    const uint32_t occ = k != kEmptyKey;
    uint32_t total;
    const uint32_t before = block_exclusive_scan256(occ, tmp, &total);
    if (threadIdx.x == 0)
      s_base = total ? atomicAdd(&st->nblocks, static_cast<unsigned long long>(total)) : 0ull;
    __syncthreads();
    if (occ) {
      bkey[s_base + before] = k;
      bslot[s_base + before] = static_cast<int32_t>(i);
      lo = k < lo ? k : lo;
      hi = k > hi ? k : hi;
    }
    __syncthreads();
  }
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    const unsigned long long h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    lo = l2 < lo ? l2 : lo;
    hi = h2 > hi ? h2 : hi;
  }
  if ((threadIdx.x & 31) == 0) {
    wlo[threadIdx.x >> 5] = lo;
    whi[threadIdx.x >> 5] = hi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) {
      lo = wlo[w] < lo ? wlo[w] : lo;
      hi = whi[w] > hi ? whi[w] : hi;
    }
    if (lo <= hi) {
      atomicMin(&st->kmin, lo);
      atomicMax(&st->kmax, hi);
    }
  }
}

// Voxels of the sorted blocks [t * 2048, (t + 1) * 2048) per block of 256 threads, eight
// consecutive blocks per thread.
constexpr int kStartTile = 2048;

__device__ __forceinline__ const int32_t* sorted_slots(const int32_t* b0, const int32_t* b1,
                                                       const KmapStatus* st) {
  return (st->plan[kMaxPasses] & 1) ? b1 : b0;
}




// The block starts in one pass (a decoupled look-back scan, as the sort passes use it): a
// block takes the next tile of 2048 sorted blocks (tile numbers from a counter, in order),
// sums their popcounts, publishes the sum, walks back over the earlier tiles' published
// values to the count before its own (every wait bounded), publishes its inclusive count
// and writes each block's first position into its slot. The last tile also records the
// number of positions and the duplicate test (every voxel valid and inserted, fewer
// distinct codes than voxels).
constexpr unsigned long long kScanTag = 15ull << 34;   // no sort pass uses this tag

__global__ void __launch_bounds__(256) kmap_h_starts(const int32_t* __restrict__ b0,
                                                     const int32_t* __restrict__ b1,
                                                     Slot* table,
                                                     unsigned long long* __restrict__ status,
                                                     int64_t N, KmapStatus* st) {
  __shared__ uint32_t tmp[8];
  __shared__ uint32_t s_tile;
  __shared__ unsigned long long s_before;
  const unsigned long long nb = st->nblocks;
  const int64_t ntile = static_cast<int64_t>((nb + kStartTile - 1) / kStartTile);
  const int32_t* bs = sorted_slots(b0, b1, st);
  constexpr int kPer = kStartTile / 256;
  for (;;) {
    if (threadIdx.x == 0) s_tile = atomicAdd(&st->scan_ctr, 1u);
    __syncthreads();
    const int64_t t = s_tile;
    if (t >= ntile) {
      if (nb == 0 && t == 0) {   // no block at all (every coordinate out of range)
        st->npos = 0;
        if (N > 0 && !(st->flags & (kFlagCoord | kFlagFull))) atomicOr(&st->flags, kFlagDup);
      }
      return;
    }
    const unsigned long long e0 = t * static_cast<unsigned long long>(kStartTile) +
                                  threadIdx.x * kPer;
    int32_t slot[kPer];
    uint32_t cnt[kPer], mine = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      slot[q] = e0 + q < nb ? bs[e0 + q] : -1;
      cnt[q] = slot[q] >= 0 ? static_cast<uint32_t>(__popcll(table[slot[q]].mask)) : 0u;
      mine += cnt[q];
    }
    uint32_t total;
    const uint32_t pre = block_exclusive_scan256(mine, tmp, &total);
    if (threadIdx.x == 0) {
      unsigned long long* my = status + t * 256;
      unsigned long long before = 0;
      if (t == 0) {
        st_relaxed_u64(my, kScanTag | kTileInclusive | total);
      } else {
        st_relaxed_u64(my, kScanTag | kTileAggregate | total);
        const unsigned long long t0 = global_timer_ns();
        for (int64_t u = t - 1; u >= 0;) {
          const unsigned long long v = ld_relaxed_u64(status + u * 256);
          if ((v & (63ull << 34)) != kScanTag || !(v & (3ull << 32))) {   // not yet published
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              atomicOr(&st->flags, kFlagInternal);
              break;
            }
            continue;
          }
          before += static_cast<uint32_t>(v);
          if ((v & (3ull << 32)) == kTileInclusive) break;
          --u;
        }
        st_relaxed_u64(my, kScanTag | kTileInclusive | (before + total));
      }
      s_before = before;
      if (t == ntile - 1) {
        const unsigned long long npos = before + total;
        st->npos = npos;
        if (npos < static_cast<unsigned long long>(N) && !(st->flags & (kFlagCoord | kFlagFull)))
          atomicOr(&st->flags, kFlagDup);
      }
    }
    __syncthreads();
    unsigned long long at = s_before + pre;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (slot[q] >= 0) table[slot[q]].start = at;
      at += cnt[q];
    }
    __syncthreads();   // s_tile and s_before are free for the next tile
  }
}

// Each voxel to its position: sort key to mk, input row to ix (and to order). Repeats of
// one coordinate share a position (one of them lands there; the build then fails), so
// the positions [0, npos) are all written.
__global__ void __launch_bounds__(256) kmap_h_scatter(
    const int4* __restrict__ coords, const uint32_t* __restrict__ slot_of, int64_t N, int bits,
    const Slot* __restrict__ table, unsigned long long* __restrict__ mk, int32_t* __restrict__ ix,
    int32_t* __restrict__ order, KmapStatus* st) {
  if (blockIdx.x == 0 && threadIdx.x == 0) st->plan[kMaxPasses] = 0;   // the probe reads mk, ix
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < N; i += stride) {
    const uint32_t h = slot_of[i];
    if (h == kSkip) continue;
    const unsigned long long key = sort_key(coords[i], bits);
    const unsigned long long mask = table[h].mask;
    const unsigned long long pos =
        table[h].start + __popcll(mask & ((1ull << (key & 63u)) - 1ull));
    if (pos < static_cast<unsigned long long>(N)) {
      mk[pos] = key;
      ix[pos] = static_cast<int32_t>(i);
      if (order) order[pos] = static_cast<int32_t>(i);
    } else {
      bad = true;
    }
  }
  if (bad) atomicOr(&st->flags, kFlagInternal);
}

// 8. ------------------------------------------------------------------------------
// Warp-cooperative probe over the sorted order. A warp takes 32 consecutive sorted
// positions, one voxel per lane. Its voxels fall into a few block runs (a run is one
// occupied 4x4x4 block); for every run the warp looks up, spread over its lanes, the 27
// blocks around the run's block, which hold every neighbour of every voxel of the run,
// and keeps their occupancy masks and first sorted positions in shared memory. Each
// lane then resolves its voxel's 27 neighbours: a table indexed by the voxel's place
// inside its block (the low 6 bits of its Morton code) gives, per offset, which of the
// 27 blocks holds the neighbour and the neighbour's bit there; a bit test and a
// popcount give the neighbour's sorted position, and the input row there is the answer.
// The rows are staged in shared memory and written out coalesced. Depending on the mode
// the warp writes
//   kProbeNbr     each voxel's row of nbr at its input row;
//   kProbeSorted  its row at its sorted position (a Morton-ordered copy of the table,
//                 which the tile plan reorders) and its 27-bit presence mask as a
//                 grouping key (window << 27 | mask) with its sorted position as the
//                 value -- or, for a plan of one-voxel windows (perm given), the plan's
//                 perm entry and the OR of the masks into the tile's offset mask.
enum ProbeMode { kProbeNbr = 0, kProbeSorted = 1 };
constexpr int kProbeThreads = 128;
constexpr int kProbeWarps = kProbeThreads / 32;
constexpr int kRunsAtOnce = 6;   // runs of a warp's 32 voxels whose blocks are held at once

// One hash lookup from slot h on, at most `probes` slots: the block's occupancy mask and
// first sorted position (0 and 0 when the block is not in the table). A slot is one
// 32-byte load.
__device__ __forceinline__ void block_lookup(const Slot* __restrict__ table,
                                             unsigned long long key, unsigned long long h,
                                          unsigned long long cmask, int probes,
                                          unsigned long long& mask, int32_t& start, bool& full) {
  mask = 0;
  start = 0;
  for (int probe = 0; probe < probes; ++probe) {
    uint32_t w[8];
    asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(table + h));
    const unsigned long long k = (static_cast<unsigned long long>(w[1]) << 32) | w[0];
    if (k == key) {
      mask = (static_cast<unsigned long long>(w[3]) << 32) | w[2];
      start = static_cast<int32_t>(w[4]);
      return;
    }
    if (k == kEmptyKey) return;
    h = (h + 1) & cmask;
  }
  full = true;
}

// Morton place (bit t of x -> 3t, y -> 3t+1, z -> 3t+2) of (z, y, x) inside a 4x4x4 block.
__host__ __device__ __forceinline__ int place_in_block(int z, int y, int x) {
  return (x & 1) | ((y & 1) << 1) | ((z & 1) << 2) | ((x & 2) << 2) | ((y & 2) << 3) |
         ((z & 2) << 4);
}

template <int MODE>
__global__ void __launch_bounds__(kProbeThreads, 7) kmap_probe(
    const unsigned long long* __restrict__ mk0, const unsigned long long* __restrict__ mk1,
    const int32_t* __restrict__ ix0, const int32_t* __restrict__ ix1, int64_t N, int res,
    int bits, const Slot* __restrict__ table, int32_t* __restrict__ nbr,
    unsigned long long* __restrict__ key2, int32_t* __restrict__ val2, int window_shift,
    int32_t* __restrict__ perm, uint32_t* __restrict__ tmask, KmapStatus* st) {
  // tbl[k][p] = (2 x which of the 27 blocks around a voxel's block holds its neighbour
  // at offset k, for a voxel at place p, + which half of that block's mask) << 5 |
  // (31 - the neighbour's bit in that half): shifted left by that amount, the half has
  // the neighbour's bit as its sign and its popcount is the neighbour's rank + 1; the
  // lanes of a warp read one offset's row at their own places, without bank conflicts
  __shared__ uint16_t tbl[27 * 64];
  // per warp: the 27 blocks of up to kRunsAtOnce runs, each as two halves {32-bit mask,
  // first position of the half - 1}, the runs' block keys, and the 32 voxels' rows
  __shared__ uint2 s_blk[kProbeWarps][kRunsAtOnce][54];
  __shared__ unsigned long long s_runkey[kProbeWarps][32];
  __shared__ uint32_t s_need[kProbeWarps][32];   // per run: the blocks its voxels reach
  // per warp: the lookups of the runs held at once, run << 5 | block (0..26), in order
  __shared__ uint8_t s_list[kProbeWarps][kRunsAtOnce * 27];
  __shared__ uint32_t need_tbl[64];              // per place: the blocks a voxel there reaches
  __shared__ __align__(16) int32_t s_row[kProbeWarps][32 * 27];
  for (int e = threadIdx.x; e < 27 * 64; e += kProbeThreads) {
    const int k = e >> 6, p = e & 63;
    const int lz = ((p >> 2) & 1) | ((p >> 4) & 2), ly = ((p >> 1) & 1) | ((p >> 3) & 2),
              lx = (p & 1) | ((p >> 2) & 2);
    const int nz = lz + k / 9 - 1, ny = ly + (k / 3) % 3 - 1, nx = lx + k % 3 - 1;
    const int kb = 9 * ((nz >> 2) + 1) + 3 * ((ny >> 2) + 1) + ((nx >> 2) + 1);
    const int np = place_in_block(nz & 3, ny & 3, nx & 3);
    tbl[e] = static_cast<uint16_t>(((2 * kb + (np >> 5)) << 5) | (31 - (np & 31)));
  }
  for (int p = threadIdx.x; p < 64; p += kProbeThreads) {
    uint32_t need = 0;
    for (int k = 0; k < 27; ++k) {
      const int lz = ((p >> 2) & 1) | ((p >> 4) & 2), ly = ((p >> 1) & 1) | ((p >> 3) & 2),
                lx = (p & 1) | ((p >> 2) & 2);
      const int nz = lz + k / 9 - 1, ny = ly + (k / 3) % 3 - 1, nx = lx + k % 3 - 1;
      need |= 1u << (9 * ((nz >> 2) + 1) + 3 * ((ny >> 2) + 1) + ((nx >> 2) + 1));
    }
    need_tbl[p] = need;
  }
  __syncthreads();
  const bool second = st->plan[kMaxPasses] & 1;
  const unsigned long long* mk = second ? mk1 : mk0;
  const int32_t* ix = second ? ix1 : ix0;
  // the positions of the order (fewer than N only when the hashed front end skipped a
  // voxel: the build then fails, and nbr is unspecified)
  if (static_cast<unsigned long long>(N) > st->npos) N = static_cast<int64_t>(st->npos);
  const unsigned long long cmask = st->cap - 1;
  const int max_probe = st->cap < kMaxProbe ? static_cast<int>(st->cap) : kMaxProbe;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  uint32_t* need_sm = s_need[wid];
  uint2 (*blk_sm)[54] = s_blk[wid];
  unsigned long long* runkey = s_runkey[wid];
  int32_t* row_sm = s_row[wid];
  // Block keys are (batch | Morton code of the block's coordinates); a neighbour block's
  // key comes from the run's by a masked increment or decrement of one axis's
  // interleaved bits, and the bounds test compares those bits, which keep the order of
  // the coordinate, with the interleaved largest block coordinate.
  const uint32_t bmax = static_cast<uint32_t>(res - 1) >> 2;
  const uint32_t ones = (1u << (bits - 2)) - 1u;
  const unsigned long long ax = spread3(ones), ay = ax << 1, az = ax << 2;
  const unsigned long long lx = spread3(bmax), ly = lx << 1, lz = lx << 2;
  const uint32_t n32 = static_cast<uint32_t>(N);
  constexpr unsigned kAll = 0xffffffffu;
  bool full = false, bad = false;
  const int64_t nwarps = (int64_t(gridDim.x) * kProbeThreads) >> 5;
  const bool want_row = MODE == kProbeNbr || perm != nullptr;
  // a round's sort key and row, loaded one round ahead
  int64_t w = (blockIdx.x * int64_t(kProbeThreads) + threadIdx.x) >> 5;
  unsigned long long m_next = ~0ull;
  int32_t orow_next = -1;
  if (w * 32 + lane < N) {
    m_next = mk[w * 32 + lane];
    if (want_row) orow_next = __ldg(ix + w * 32 + lane);
  }
  for (; w * 32 < N; w += nwarps) {
    if (MODE == kProbeSorted) {   // the previous rows' bulk copy has read the staging rows
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
    }
    const int64_t s = w * 32 + lane;
    const bool valid = s < N;
    const int nvalid = (N - w * 32) < 32 ? static_cast<int>(N - w * 32) : 32;
    const unsigned long long m = m_next;
    const unsigned long long blk = m >> 6;
    const int32_t orow = orow_next;   // the row this lane's voxel is written to
    {
      const int64_t sn = s + nwarps * 32;
      m_next = ~0ull;
      orow_next = -1;
      if (sn < N) {
        m_next = mk[sn];
        if (want_row) orow_next = __ldg(ix + sn);
      }
    }
    const unsigned long long prev = __shfl_up_sync(kAll, blk, 1);
    const unsigned newb = __ballot_sync(kAll, valid && (lane == 0 || prev != blk));
    const int run = __popc(newb & ((2u << lane) - 1u)) - 1;   // this lane's run, from 0
    const int nruns = __popc(newb);
    if ((newb >> lane) & 1u) {
      runkey[run] = blk;
      need_sm[run] = 0;
    }
    __syncwarp();
    const uint32_t p = static_cast<uint32_t>(m) & 63u;
    if (valid) atomicOr(&need_sm[run], need_tbl[p]);
    __syncwarp();
    uint32_t present_mask = 0;
    for (int g0 = 0; g0 < nruns; g0 += kRunsAtOnce) {
      const int G = nruns - g0 < kRunsAtOnce ? nruns - g0 : kRunsAtOnce;
      // the blocks these runs' voxels reach (of the 27 around each run's block), listed
      // run by run (lane kb < 27 places block kb of run r at its rank), then looked up
      // one per lane
      uint8_t* list = s_list[wid];
      int total = 0;
      for (int r = 0; r < G; ++r) {
        const uint32_t nm = need_sm[g0 + r];
        if (lane < 27 && ((nm >> lane) & 1u))
          list[total + __popc(nm & ((1u << lane) - 1u))] = static_cast<uint8_t>((r << 5) | lane);
        total += __popc(nm);
      }
      __syncwarp();
      // a lane's lookups go kLookups at a time, their first slots loaded together (a
      // further probe, after a collision, is rare)
      constexpr int kLookups = 2;
      for (int q0 = 0; q0 < total; q0 += 32 * kLookups) {
        unsigned long long key[kLookups];
        bool use[kLookups];
        int ent[kLookups];
        uint4 first[kLookups];
        uint32_t first_start[kLookups];
#pragma unroll
        for (int u = 0; u < kLookups; ++u) {
          const int q = q0 + 32 * u + lane;
          ent[u] = q < total ? list[q] : -1;
          key[u] = 0;
          use[u] = false;
          if (ent[u] >= 0) {
            const int kb = ent[u] & 31;
            const int dz = kb / 9 - 1, dy = (kb / 3) % 3 - 1, dx = kb % 3 - 1;
            unsigned long long k = runkey[g0 + (ent[u] >> 5)];
            bool inside = true;
            if (dx > 0) { inside &= (k & ax) < lx; k = (((k | ~ax) + 1) & ax) | (k & ~ax); }
            if (dx < 0) { inside &= (k & ax) != 0; k = (((k & ax) - 1) & ax) | (k & ~ax); }
            if (dy > 0) { inside &= (k & ay) < ly; k = (((k | ~ay) + 1) & ay) | (k & ~ay); }
            if (dy < 0) { inside &= (k & ay) != 0; k = (((k & ay) - 1) & ay) | (k & ~ay); }
            if (dz > 0) { inside &= (k & az) < lz; k = (((k | ~az) + 1) & az) | (k & ~az); }
            if (dz < 0) { inside &= (k & az) != 0; k = (((k & az) - 1) & az) | (k & ~az); }
            key[u] = k;
            use[u] = inside;
          }
        }
#pragma unroll
        for (int u = 0; u < kLookups; ++u) {
          if (use[u]) {
            const Slot* sl = table + (mix64(key[u]) & cmask);
            first[u] = __ldg(reinterpret_cast<const uint4*>(sl));   // key, mask
            first_start[u] = __ldg(reinterpret_cast<const uint32_t*>(&sl->start));
          }
        }
#pragma unroll
        for (int u = 0; u < kLookups; ++u) {
          if (ent[u] < 0) continue;
          unsigned long long bm = 0;
          int32_t bb = 0;
          if (use[u]) {
            const unsigned long long k =
                (static_cast<unsigned long long>(first[u].y) << 32) | first[u].x;
            if (k == key[u]) {
              bm = (static_cast<unsigned long long>(first[u].w) << 32) | first[u].z;
              bb = static_cast<int32_t>(first_start[u]);
            } else if (k != kEmptyKey) {
              block_lookup(table, key[u], (mix64(key[u]) + 1) & cmask, cmask, max_probe - 1,
                           bm, bb, full);
            }
          }
          const int r = ent[u] >> 5, kb = ent[u] & 31;
          const uint32_t lo = static_cast<uint32_t>(bm), hi = static_cast<uint32_t>(bm >> 32);
          blk_sm[r][2 * kb] = make_uint2(lo, static_cast<uint32_t>(bb) - 1u);
          blk_sm[r][2 * kb + 1] = make_uint2(hi, static_cast<uint32_t>(bb) + __popc(lo) - 1u);
        }
      }
      __syncwarp();
      if (valid && run >= g0 && run < g0 + G) {   // this lane's voxel: its 27 neighbours
        const uint2* nb = blk_sm[run - g0];
#pragma unroll
        for (int k = 0; k < 27; ++k) {
          const uint32_t e = tbl[k * 64 + p];
          const uint2 half = nb[e >> 5];   // {mask half, its first position - 1}
          const uint32_t t = __funnelshift_l(0u, half.x, e);   // half.x << (e & 31)
          int32_t val = -1;
          if (static_cast<int32_t>(t) < 0) {   // the neighbour's bit
            const uint32_t pos = half.y + __popc(t);
            present_mask |= 1u << k;
            if (pos < n32) val = __ldg(ix + pos);
            else bad = true;
          }
          row_sm[lane * 27 + k] = val;
        }
      }
      __syncwarp();
    }
    // the 32 rows, out of shared memory
    if (MODE == kProbeSorted) {   // contiguous: rows of consecutive sorted positions
      int32_t* dst = nbr + w * 32 * 27;   // 3456 bytes per warp: 16-byte aligned
      // one bulk copy of the staged rows (whole 16-byte pieces; the copy engine writes
      // them while the warp goes on, and the next round waits only for it to have read
      // the staging rows), the ragged tail of a partial warp by plain stores
      const int nw = nvalid * 27, n4 = nw >> 2;
      fence_proxy_async_smem();   // the lanes' row writes before the copy reads them
      __syncwarp();
      if (lane == 0 && n4 > 0) {
        bulk_store(dst, smem_u32(row_sm), static_cast<uint32_t>(n4) * 16u);
        bulk_commit();
      }
      for (int i = 4 * n4 + lane; i < nw; i += 32) __stcs(dst + i, row_sm[i]);
      if (perm) {   // a window-1 plan: perm and the tile's offset mask directly
        if (valid) perm[s] = orow;
        const uint32_t m = __reduce_or_sync(kAll, present_mask);
        if (lane == 0) atomicOr(tmask + (w >> 2), m | (1u << 13));   // 4 warps per tile
      } else if (valid) {
        key2[s] = (static_cast<unsigned long long>(s >> window_shift) << 27) | present_mask;
        val2[s] = static_cast<int32_t>(s);
      }
    } else {                      // row by row, each to its input row
      for (int j = 0; j < nvalid; ++j) {
        const uint32_t r = static_cast<uint32_t>(__shfl_sync(kAll, orow, j));
        if (lane < 27 && r < n32) __stcs(nbr + static_cast<size_t>(r) * 27u + lane, row_sm[j * 27 + lane]);
      }
    }
    __syncwarp();
  }
  if (MODE == kProbeSorted && lane == 0) bulk_wait_all();   // every row written
  if (__any_sync(kAll, full) && lane == 0) atomicOr(&st->flags, kFlagFull);
  if (__any_sync(kAll, bad) && lane == 0) atomicOr(&st->flags, kFlagInternal);
}

// The tile plan from the grouping sort, a block of 128 threads per tile: plan row r is
// the voxel at sorted position s = v2[r] (grouping key k2[r] = window << 27 | mask);
// perm[r] = its input row, its row of the plan's nbr is the Morton-ordered row s
// (copied: 27 contiguous words read, the tile's 128 rows written as one stretch), and
// the tile's offset mask is the OR of its rows' presence masks (the centre always
// included).
__global__ void __launch_bounds__(128) kmap_plan_index(
    const unsigned long long* __restrict__ k2a, const unsigned long long* __restrict__ k2b,
    const int32_t* __restrict__ v2a, const int32_t* __restrict__ v2b,
    const int32_t* __restrict__ ix0, const int32_t* __restrict__ ix1, int64_t N, int64_t ntiles,
    const int32_t* __restrict__ nbr_sorted, int32_t* __restrict__ perm,
    int32_t* __restrict__ pnbr, uint32_t* __restrict__ tmask, KmapStatus* st) {
  const bool sec2 = st->plan2[kMaxPasses] & 1;
  const unsigned long long* k2 = sec2 ? k2b : k2a;
  const int32_t* v2 = sec2 ? v2b : v2a;
  const int32_t* ix = (st->plan[kMaxPasses] & 1) ? ix1 : ix0;
  __shared__ uint32_t wm[4];
  __shared__ int32_t src[128];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  bool bad = false;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t r = t * 128 + threadIdx.x;
    uint32_t m = 0;
    int32_t sp = -1;
    if (r < N) {
      sp = v2[r];
      if (static_cast<uint64_t>(sp) < static_cast<uint64_t>(N)) {
        perm[r] = ix[sp];
        m = static_cast<uint32_t>(k2[r]) & 0x7FFFFFFu;
      } else {
        perm[r] = -1;
        sp = -1;
        bad = true;
      }
    }
    src[threadIdx.x] = sp;
    for (int o = 16; o > 0; o >>= 1) m |= __shfl_xor_sync(0xffffffffu, m, o);
    if (lane == 0) wm[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) tmask[t] = wm[0] | wm[1] | wm[2] | wm[3] | (1u << 13);
    const int rows = static_cast<int>((N - t * 128) < 128 ? (N - t * 128) : 128);
    int32_t* dst = pnbr + t * 128 * 27;
    for (int w = threadIdx.x; w < rows * 27; w += 128) {
      const int rr = w / 27, k = w - 27 * rr;
      const int32_t from = src[rr];
      dst[w] = from >= 0 ? nbr_sorted[int64_t(from) * 27 + k] : -1;
    }
    __syncthreads();
  }
  if (bad) atomicOr(&st->flags, kFlagInternal);
}

// Folds the build's status into the device error word (asynchronous builds).
__global__ void kmap_report(const KmapStatus* st, int* err) {
  const int f = st->flags;
  int bits = 0;
  if (f & kFlagCoord) bits |= kDevErrKmapCoord;
  if (f & kFlagDup) bits |= kDevErrKmapDup;
  if (f & kFlagFull) bits |= kDevErrKmapFull;
  if (f & kFlagInternal) bits |= kDevErrKmapInternal;
  if (bits) atomicOr(err, bits);
}

int grid_for(int64_t work, int threads, int per_sm) {
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = int64_t(num_sms()) * per_sm;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

// Validate + pack (Morton keys, batch above them) and the stable LSD radix sort of
// (key, input row), shared by the kernel map and the downsample. Leaves the status
// word's plan saying which of (mk0, ix0) / (mk1, ix1) holds the sorted result.
// Stage timing of the kernel-map builds (subm3d_kmap_stage_timing): while enabled on a
// host thread, each build on that thread records a CUDA event on its stream before its
// first stage and after each stage, so that subm3d_kmap_stage_times can report the GPU
// time of every stage of the last build. Off by default; recording events adds no
// synchronisation.
struct StageTimer {
  static constexpr int kMax = 40;
  bool on = false;
  int n = 0;
  cudaEvent_t ev[kMax] = {};
  const char* name[kMax] = {};
  void begin(cudaStream_t stream) {
    n = 0;
    mark("start", stream);
  }
  void mark(const char* what, cudaStream_t stream) {
    if (!on || n >= kMax) return;
    if (!ev[n] && cudaEventCreate(&ev[n]) != cudaSuccess) return;
    if (cudaEventRecord(ev[n], stream) != cudaSuccess) return;
    name[n++] = what;
  }
};
thread_local StageTimer g_stage;

// The count / scan / scatter passes of a stable LSD radix sort of (u64 key, i32 value)
// pairs ping-ponging between (k0, v0) and (k1, v1); plans[p] (device) says whether pass p
// runs and which buffer it reads, plans[kMaxPasses] which one holds the result.
// count: when not NULL, the number of pairs is read on the device (at most N).
// small_tiles: 512-key tiles (the scratch holds status words for that many tiles).
int launch_radix(unsigned long long* k0, unsigned long long* k1, int32_t* v0, int32_t* v1,
                 int64_t N, int npass, uint32_t* hist, char* scratch, int64_t nblk,
                 const int* plans, KmapStatus* st, cudaStream_t stream,
                 const char* stage = "sort pass", const unsigned long long* count = nullptr,
                 bool small_tiles = false) {
  static PerDevice<bool> attr_set[2];
  const int arc0 = set_smem_limit_once(attr_set[0],
                                       reinterpret_cast<const void*>(kmap_onesweep<kSortItems>),
                                       scatter_smem(kSortTile), "kmap_onesweep");
  if (arc0 != SUBM3D_OK) return arc0;
  const int arc1 = set_smem_limit_once(
      attr_set[1], reinterpret_cast<const void*>(kmap_onesweep<kBlockSortItems>),
      scatter_smem(kSortThreads * kBlockSortItems), "kmap_onesweep");
  if (arc1 != SUBM3D_OK) return arc1;
  const int64_t ntile = small_tiles ? nblk * kSmallTileRatio : nblk;
  const SortScratch S = sort_scratch(scratch, ntile);
  kmap_hist<<<grid_for(N, 256, 4), 256, 0, stream>>>(
      k0, N, count, npass, plans, hist, S, ntile,
      small_tiles ? kSortThreads * kBlockSortItems : kSortTile);
  SUBM3D_LAUNCHED("kmap_hist");
  kmap_digit_starts<<<1, 256, 0, stream>>>(hist, npass, S);
  SUBM3D_LAUNCHED("kmap_digit_starts");
  g_stage.mark("digit histograms", stream);
  // the blocks that fit on the GPU at once (each takes tiles until none are left)
  static PerDevice<int> fit[2];
  int per_sm = 0;
  {
    const int which = small_tiles ? 1 : 0;
    const int rc = fit[which].get(&per_sm, [which](int* v) -> int {
      int n = 0;
      const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n,
          which ? reinterpret_cast<const void*>(kmap_onesweep<kBlockSortItems>)
                : reinterpret_cast<const void*>(kmap_onesweep<kSortItems>),
          kSortThreads,
          which ? scatter_smem(kSortThreads * kBlockSortItems) : scatter_smem(kSortTile));
      *v = (e == cudaSuccess && n > 0) ? n : 1;
      return static_cast<int>(SUBM3D_OK);
    });
    if (rc != SUBM3D_OK) return rc;
  }
  const int64_t resident = int64_t(num_sms()) * per_sm;
  const int grid = static_cast<int>(ntile < resident ? ntile : resident);
  for (int p = 0; p < npass; ++p) {
    if (small_tiles)
      kmap_onesweep<kBlockSortItems>
          <<<grid, kSortThreads, scatter_smem(kSortThreads * kBlockSortItems), stream>>>(
              k0, k1, v0, v1, N, count, p, ntile, plans, S, st);
    else
      kmap_onesweep<kSortItems><<<grid, kSortThreads, scatter_smem(kSortTile), stream>>>(
          k0, k1, v0, v1, N, count, p, ntile, plans, S, st);
    SUBM3D_LAUNCHED("kmap_onesweep");
    g_stage.mark(stage, stream);
  }
  return SUBM3D_OK;
}

int launch_sort(const int4* c4, int64_t N, int32_t res, const Layout& L, char* ws,
                cudaStream_t stream) {
  KmapStatus* st = reinterpret_cast<KmapStatus*>(ws + L.status);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  unsigned long long* mk0 = reinterpret_cast<unsigned long long*>(ws + L.mk0);
  unsigned long long* mk1 = reinterpret_cast<unsigned long long*>(ws + L.mk1);
  int32_t* ix0 = reinterpret_cast<int32_t*>(ws + L.ix0);
  int32_t* ix1 = reinterpret_cast<int32_t*>(ws + L.ix1);
  int bits = 2;   // at least one whole 4x4x4 block level below the batch bits
  while ((1 << bits) < res) ++bits;
  const int npass = (3 * bits + 16 + 7) / 8;
  uint32_t* hist2 = L.hist2 ? reinterpret_cast<uint32_t*>(ws + L.hist2) : nullptr;
  kmap_init<<<8, 256, 0, stream>>>(st, hist, hist2);
  SUBM3D_LAUNCHED("kmap_init");
  kmap_pack<<<grid_for(N, 256, 4), 256, 0, stream>>>(c4, N, res, bits, mk0, ix0, st);
  SUBM3D_LAUNCHED("kmap_pack");
  kmap_plan<<<1, 1, 0, stream>>>(npass, N, st);
  SUBM3D_LAUNCHED("kmap_plan");
  g_stage.mark("pack", stream);
  const int* plans = reinterpret_cast<const int*>(reinterpret_cast<const char*>(st) +
                                                  offsetof(KmapStatus, plan));
  return launch_radix(mk0, mk1, ix0, ix1, N, npass, hist, ws + L.cnt, L.nblk, plans, st, stream);
}

// SparseDownsample(2) / SparseUpsample(2) ------------------------------------------
// ("pixal3d_mrp_mlx README", scope table "Scope, measured against the shared core": a
// downsample with a pooling mode, and the upsample as its cache-paired inverse that
// reuses the stored subdivision.)
// The parent of a fine voxel (b, z, y, x) is (b, z>>1, y>>1, x>>1). Its sort key is the
// fine key >> 3 (the lowest Morton triple is the place inside the 2x2x2 cell), so in the
// sorted order each parent's children are adjacent and parents come in (batch, Morton)
// order. A parent starts where key >> 3 changes; a scan over 2048-position tiles numbers
// the parents.

constexpr int kDsTile = kSortTile;   // sorted positions per tile (256 threads x 8)

struct DsLayout {
  Layout k;              // status, histograms and sort buffers (no hash table)
  size_t tsum;           // uint32 [ntile + 1]: parents before each tile, then M
  size_t pstart;         // int32 [N + 1]: first sorted position of each parent, then N
  size_t total;
  int64_t ntile;
};

DsLayout make_ds_layout(int64_t N) {
  DsLayout D;
  D.k = make_layout(N, 0);
  D.ntile = (N + kDsTile - 1) / kDsTile;
  size_t o = D.k.total;
  D.tsum = o;   o = align256(o + sizeof(uint32_t) * (D.ntile + 1));
  D.pstart = o; o = align256(o + sizeof(int32_t) * (N + 1));
  D.total = o;
  return D;
}

__device__ __forceinline__ bool parent_starts(const unsigned long long* mk, int64_t s) {
  return s == 0 || (mk[s - 1] >> 3) != (mk[s] >> 3);
}

// The sort keys of a voxel set in a Morton order the caller already has (the kernel
// map's `order` on the same coordinates): mk[s] = key of input row order[s]. Checks what
// the sort would otherwise guarantee: rows in range, coordinates in range, keys
// ascending (an order that is not the Morton order is an argument error).
__global__ void __launch_bounds__(256) ds_keys_in_order(
    const int4* __restrict__ coords, const int32_t* __restrict__ order, int64_t N, int res,
    int bits, unsigned long long* __restrict__ mk, int32_t* __restrict__ ix, KmapStatus* st) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31;
  auto key_of = [&](int32_t r, bool& good) -> unsigned long long {
    const int4 c = coords[r];
    good = good && static_cast<unsigned>(c.x) <= SUBM3D_MAX_BATCH &&
           static_cast<unsigned>(c.y) < static_cast<unsigned>(res) &&
           static_cast<unsigned>(c.z) < static_cast<unsigned>(res) &&
           static_cast<unsigned>(c.w) < static_cast<unsigned>(res);
    return (static_cast<unsigned long long>(c.x) << (3 * bits)) | morton3(c.y, c.z, c.w);
  };
  // whole warps per round: the previous position's key comes from the lane before
  for (int64_t w0 = blockIdx.x * int64_t(blockDim.x) + threadIdx.x - lane; w0 < N; w0 += stride) {
    const int64_t s = w0 + lane;
    const bool live = s < N;
    const int32_t row = live ? order[s] : 0;
    unsigned long long key = 0;
    bool ok = live && static_cast<uint64_t>(row) < static_cast<uint64_t>(N);
    if (ok) key = key_of(row, ok);
    unsigned long long prev_key = __shfl_up_sync(0xffffffffu, key, 1);
    bool prev_ok = __shfl_up_sync(0xffffffffu, ok, 1);
    if (lane == 0 && s > 0 && live) {
      const int32_t prow = order[s - 1];
      prev_ok = static_cast<uint64_t>(prow) < static_cast<uint64_t>(N);
      if (prev_ok) prev_key = key_of(prow, prev_ok);
    }
    if (!live) continue;
    if (ok && s > 0 && prev_ok && prev_key > key) ok = false;
    if (!ok) {
      atomicOr(&st->flags, kFlagOrder);
      atomicMin(&st->bad_row, static_cast<long long>(s));
      key = 0;
    }
    mk[s] = key;
    ix[s] = ok ? row : 0;
  }
}

// Parents per tile; duplicate keys (adjacent equal) and sort indices out of range are
// flagged in the status word.
__global__ void __launch_bounds__(kSortThreads) ds_count(
    const unsigned long long* __restrict__ mk0, const unsigned long long* __restrict__ mk1,
    const int32_t* __restrict__ ix0, const int32_t* __restrict__ ix1, int64_t N,
    uint32_t* __restrict__ tsum, KmapStatus* st) {
  const bool second = st->plan[kMaxPasses] & 1;
  const unsigned long long* mk = second ? mk1 : mk0;
  const int32_t* ix = second ? ix1 : ix0;
  const int64_t base = blockIdx.x * int64_t(kDsTile);
  uint32_t heads = 0;
  for (int r = 0; r < kSortItems; ++r) {
    const int64_t s = base + r * kSortThreads + threadIdx.x;
    if (s >= N) break;
    const int32_t row = ix[s];
    if (static_cast<uint64_t>(row) >= static_cast<uint64_t>(N)) atomicOr(&st->flags, kFlagInternal);
    if (parent_starts(mk, s)) ++heads;
    if (s > 0 && mk[s - 1] == mk[s]) {
      atomicOr(&st->flags, kFlagDup);
      atomicMin(&st->bad_row, static_cast<long long>(row));
    }
  }
  __shared__ uint32_t tmp[8];
  uint32_t total;
  block_exclusive_scan256(heads, tmp, &total);
  if (threadIdx.x == 0) tsum[blockIdx.x] = total;
}

// One block: exclusive scan of the per-tile counts; tsum[ntile] and nblocks get M.
__global__ void __launch_bounds__(256) ds_scan(uint32_t* __restrict__ tsum, int64_t ntile,
                                               KmapStatus* st) {
  __shared__ uint32_t tmp[8];
  uint32_t carry = 0;
  for (int64_t b0 = 0; b0 < ntile; b0 += 256) {
    const int64_t b = b0 + threadIdx.x;
    const uint32_t x = b < ntile ? tsum[b] : 0u;
    uint32_t sum;
    const uint32_t pre = block_exclusive_scan256(x, tmp, &sum);
    if (b < ntile) tsum[b] = carry + pre;
    carry += sum;
  }
  if (threadIdx.x == 0) {
    tsum[ntile] = carry;
    st->nblocks = carry;
  }
}

// Each thread takes 8 consecutive sorted positions of its tile: the parent index of a
// position is the number of parent starts before it (tile offset + block scan + own
// run). Writes parent[row] for every fine row and, at each start, the parent's
// coordinates, its first sorted position and its child mask (the run is at most the
// 8 cells of a 2x2x2 block when there are no duplicates; the loop never looks further).
__global__ void __launch_bounds__(kSortThreads) ds_emit(
    const int4* __restrict__ coords, const unsigned long long* __restrict__ mk0,
    const unsigned long long* __restrict__ mk1, const int32_t* __restrict__ ix0,
    const int32_t* __restrict__ ix1, int64_t N, const uint32_t* __restrict__ tsum,
    int4* __restrict__ coarse, int32_t* __restrict__ parent, uint8_t* __restrict__ cmask,
    int32_t* __restrict__ pstart, int bits, const KmapStatus* st) {
  if (st->flags & kFlagInternal) return;
  const bool second = st->plan[kMaxPasses] & 1;
  const unsigned long long* mk = second ? mk1 : mk0;
  const int32_t* ix = second ? ix1 : ix0;
  const int64_t s0 = blockIdx.x * int64_t(kDsTile) + threadIdx.x * int64_t(kSortItems);
  // this thread's keys, and the one before them, read once
  unsigned long long kk[kSortItems + 1];
  kk[0] = s0 > 0 && s0 - 1 < N ? mk[s0 - 1] : ~0ull;
#pragma unroll
  for (int j = 0; j < kSortItems; ++j) kk[j + 1] = s0 + j < N ? mk[s0 + j] : ~0ull;
  uint32_t heads = 0;   // bit j: position s0 + j starts a parent
#pragma unroll
  for (int j = 0; j < kSortItems; ++j)
    if (s0 + j < N && (s0 + j == 0 || (kk[j] >> 3) != (kk[j + 1] >> 3))) heads |= 1u << j;
  __shared__ uint32_t tmp[8];
  uint32_t total;
  const uint32_t pre = block_exclusive_scan256(__popc(heads), tmp, &total);
  int64_t p = int64_t(tsum[blockIdx.x]) + pre - 1;   // parent of the position before s0
#pragma unroll
  for (int j = 0; j < kSortItems; ++j) {
    const int64_t s = s0 + j;
    if (s >= N) break;
    const bool head = (heads >> j) & 1u;
    if (head) ++p;
    const int32_t row = ix[s];
    parent[row] = static_cast<int32_t>(p);
    if (head) {
      // the parent's coordinates and the children's bits from the sort keys (the lowest
      // Morton triple is (z&1)<<2 | (y&1)<<1 | (x&1), the child bit)
      const unsigned long long k0 = kk[j + 1];
      const unsigned long long morton = k0 & ((1ull << (3 * bits)) - 1ull);
      coarse[p] = make_int4(static_cast<int>(k0 >> (3 * bits)),
                            static_cast<int>(compact3(morton >> 2) >> 1),
                            static_cast<int>(compact3(morton >> 1) >> 1),
                            static_cast<int>(compact3(morton) >> 1));
      pstart[p] = static_cast<int32_t>(s);
      const unsigned long long key = k0 >> 3;
      uint32_t mask = 0;
      for (int t = 0; t < 8 && s + t < N; ++t) {
        const unsigned long long kt = mk[s + t];
        if ((kt >> 3) != key) break;
        mask |= 1u << (kt & 7u);
      }
      cmask[p] = static_cast<uint8_t>(mask);
    }
    if (s == N - 1) pstart[p + 1] = static_cast<int32_t>(N);
  }
}

template <typename T, int V>
struct Vec;
template <>
struct Vec<float, 1> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[1]) { v[0] = __ldg(p); }
  static __device__ __forceinline__ void store(float* p, const float (&v)[1]) { *p = v[0]; }
};
template <>
struct Vec<float, 4> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16, 1> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[1]) {
    v[0] = __bfloat162float(__ldg(p));
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[1]) {
    *p = __float2bfloat16_rn(v[0]);
  }
};
template <>
struct Vec<__nv_bfloat16, 8> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      v[2 * e] = f.x;
      v[2 * e + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      w[e] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Pools each parent's children: a thread per (parent, V consecutive channels), fp32
// accumulation, mean = sum / count, rounded once to the feature dtype. The number of
// parents and the sorted order are read on the device (the launch is enqueued before
// the host learns M).
template <typename T, int V>
__global__ void __launch_bounds__(256) ds_pool(const T* __restrict__ feats, int C,
                                               const int32_t* __restrict__ ix0,
                                               const int32_t* __restrict__ ix1,
                                               const int32_t* __restrict__ pstart,
                                               const uint32_t* __restrict__ m_dev, int mode,
                                               T* __restrict__ out, const KmapStatus* st) {
  if (st->flags) return;   // the structure failed: the call reports it, nothing to pool
  const int32_t* ix = (st->plan[kMaxPasses] & 1) ? ix1 : ix0;
  const int64_t M = *m_dev;
  const int cv = C / V;
  const int64_t total = M * cv;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += stride) {
    const int64_t p = e / cv;
    const int c0 = static_cast<int>(e - p * cv) * V;
    const int32_t a = pstart[p], b = pstart[p + 1];
    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] = mode == SUBM3D_POOL_MAX ? -INFINITY : 0.f;
    for (int32_t s = a; s < b; s += 2) {   // two children in flight per round
      const bool two = s + 1 < b;
      const int32_t r0 = ix[s], r1 = two ? ix[s + 1] : 0;
      float v[V], u[V];
      Vec<T, V>::load(feats + int64_t(r0) * C + c0, v);
      if (two) Vec<T, V>::load(feats + int64_t(r1) * C + c0, u);
#pragma unroll
      for (int k = 0; k < V; ++k) {
        acc[k] = mode == SUBM3D_POOL_MAX ? fmaxf(acc[k], v[k]) : acc[k] + v[k];
        if (two) acc[k] = mode == SUBM3D_POOL_MAX ? fmaxf(acc[k], u[k]) : acc[k] + u[k];
      }
    }
    if (mode == SUBM3D_POOL_MEAN) {
      const float n = static_cast<float>(b - a);
#pragma unroll
      for (int k = 0; k < V; ++k) acc[k] = acc[k] / n;
    }
    Vec<T, V>::store(out + p * C + c0, acc);
  }
}

// fine[i, :] = coarse[parent[i], :]; a parent outside [0, M) gives a zero row and sets
// the device error word.
template <typename T, int V>
__global__ void __launch_bounds__(256) us_gather(const T* __restrict__ coarse, int64_t M, int C,
                                                 const int32_t* __restrict__ parent, int64_t N,
                                                 T* __restrict__ fine, int* err) {
  const int cv = C / V;
  const int64_t total = N * cv;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += stride) {
    const int64_t i = e / cv;
    const int c0 = static_cast<int>(e - i * cv) * V;
    const int32_t p = parent[i];
    float v[V];
    if (p >= 0 && p < M) {
      Vec<T, V>::load(coarse + int64_t(p) * C + c0, v);
    } else {
      if (c0 == 0) atomicOr(err, kDevErrBadParent);
#pragma unroll
      for (int k = 0; k < V; ++k) v[k] = 0.f;
    }
    Vec<T, V>::store(fine + i * C + c0, v);
  }
}

// SparseSpatial2Channel(2), the sparse pixel-unshuffle of the same scope table, on the
// downsample's subdivision: fine row i's C values go to out[parent[i], k C .. k C + C)
// with k its child bit; s2c_zero fills the blocks of absent children. The two kernels
// write disjoint bytes.
__device__ __forceinline__ int child_of(const int4 d) {   // d = (b, z, y, x)
  return ((d.y & 1) << 2) | ((d.z & 1) << 1) | (d.w & 1);
}

template <typename T, int V>
__global__ void __launch_bounds__(256) s2c_scatter(const T* __restrict__ feats,
                                                   const int4* __restrict__ coords,
                                                   const int32_t* __restrict__ parent, int64_t N,
                                                   int64_t M, int C, T* __restrict__ out, int* err) {
  const int cv = C / V;
  const int64_t total = N * cv;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += stride) {
    const int64_t i = e / cv;
    const int c0 = static_cast<int>(e - i * cv) * V;
    const int32_t p = parent[i];
    if (p < 0 || p >= M) {
      if (c0 == 0) atomicOr(err, kDevErrBadParent);
      continue;
    }
    float v[V];
    Vec<T, V>::load(feats + i * C + c0, v);
    Vec<T, V>::store(out + (int64_t(p) * 8 + child_of(coords[i])) * C + c0, v);
  }
}

template <typename T, int V>
__global__ void __launch_bounds__(256) s2c_zero(const uint8_t* __restrict__ mask, int64_t M, int C,
                                                T* __restrict__ out) {
  const int cv = C / V;
  const int64_t total = M * 8 * cv;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += stride) {
    const int64_t pk = e / cv;   // parent * 8 + child
    if ((mask[pk >> 3] >> (pk & 7)) & 1) continue;
    const int c0 = static_cast<int>(e - pk * cv) * V;
    float v[V];
#pragma unroll
    for (int k = 0; k < V; ++k) v[k] = 0.f;
    Vec<T, V>::store(out + pk * C + c0, v);
  }
}

// channel2spatial: fine[i, :] = coarse[parent[i], k C .. k C + C), k = child bit of i; a
// parent outside [0, M) gives a zero row and sets the device error word.
template <typename T, int V>
__global__ void __launch_bounds__(256) c2s_gather(const T* __restrict__ coarse,
                                                  const int4* __restrict__ coords,
                                                  const int32_t* __restrict__ parent, int64_t N,
                                                  int64_t M, int C, T* __restrict__ fine, int* err) {
  const int cv = C / V;
  const int64_t total = N * cv;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += stride) {
    const int64_t i = e / cv;
    const int c0 = static_cast<int>(e - i * cv) * V;
    const int32_t p = parent[i];
    float v[V];
    if (p >= 0 && p < M) {
      Vec<T, V>::load(coarse + (int64_t(p) * 8 + child_of(coords[i])) * C + c0, v);
    } else {
      if (c0 == 0) atomicOr(err, kDevErrBadParent);
#pragma unroll
      for (int k = 0; k < V; ++k) v[k] = 0.f;
    }
    Vec<T, V>::store(fine + i * C + c0, v);
  }
}

}  // namespace

int64_t default_hash_capacity(int64_t N) {
  int64_t cap = 64;
  while (cap < 2 * N) cap <<= 1;
  return cap;
}

size_t kmap_workspace_bytes(int64_t N, int64_t hash_capacity) {
  if (N < 0) return 0;
  const int64_t cap = hash_capacity > 0 ? hash_capacity : default_hash_capacity(N);
  return make_layout(N, cap).total;
}

namespace {

// The steps every kernel-map build shares (validate + pack, Morton sort, block runs,
// table, insert) followed by the probe for `nbr` (input order), or, when `plan` is
// given, by the tile plan's steps: presence masks in sorted order, the grouping sort,
// the plan's index arrays and the probe that writes the plan's rows. With `sync` the
// call waits for the stream and returns the device-side status; without it the status
// is folded into the device error word (read by subm3d_forward_status) and nothing
// waits.
int kmap_run(const char* fn, const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
             int32_t* order, int64_t hash_capacity, int64_t window, void* plan,
             size_t plan_bytes, void* workspace, size_t ws_bytes, bool sync,
             cudaStream_t stream, bool force_sorted = false) {
  const bool grouped = plan != nullptr;
  if (N < 0 || N > 0x7FFFFFFFll) {
    set_error("%s: N=%lld outside [0, 2^31)", fn, (long long)N);
    return SUBM3D_ERR_ARG;
  }
  if (res < 1 || res > SUBM3D_MAX_RES) {
    set_error("%s: res=%d outside [1, %d]", fn, res, SUBM3D_MAX_RES);
    return SUBM3D_ERR_ARG;
  }
  if (hash_capacity != 0 && (hash_capacity < 8 || (hash_capacity & (hash_capacity - 1)) ||
                             hash_capacity > (int64_t(1) << 40))) {
    set_error("%s: hash_capacity=%lld is not 0 or a power of two in [8, 2^40]", fn,
              (long long)hash_capacity);
    return SUBM3D_ERR_ARG;
  }
  if (grouped && (window < 1 || window > (int64_t(1) << 30) || (window & (window - 1)))) {
    set_error("%s: window=%lld is not a power of two in [1, 2^30]", fn, (long long)window);
    return SUBM3D_ERR_ARG;
  }
  if (N == 0) return SUBM3D_OK;
  if (!coords || (!grouped && !nbr) || !workspace) {
    set_error("%s: NULL pointer (coords=%p nbr=%p plan=%p workspace=%p)", fn, (const void*)coords,
              (void*)nbr, plan, workspace);
    return SUBM3D_ERR_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(coords) & 15) || (reinterpret_cast<uintptr_t>(nbr) & 15) ||
      (order && (reinterpret_cast<uintptr_t>(order) & 15)) ||
      (reinterpret_cast<uintptr_t>(plan) & 255)) {
    set_error("%s: coords=%p nbr=%p order=%p must be 16-byte aligned and plan=%p 256-byte aligned",
              fn, (const void*)coords, (void*)nbr, (void*)order, plan);
    return SUBM3D_ERR_ARG;
  }
  const PlanLayout PL = plan_layout(N);
  if (grouped && plan_bytes < PL.total) {
    set_error("%s: plan of %zu bytes, need %zu for N=%lld", fn, plan_bytes, PL.total, (long long)N);
    return SUBM3D_ERR_ARG;
  }
  const int64_t cap_max = hash_capacity > 0 ? hash_capacity : default_hash_capacity(N);
  const Layout L = make_layout(N, cap_max, grouped);
  if (reinterpret_cast<uintptr_t>(workspace) & 255) {
    set_error("%s: workspace=%p must be 256-byte aligned", fn, workspace);
    return SUBM3D_ERR_WORKSPACE;
  }
  if (ws_bytes < L.total) {
    set_error("%s: workspace of %zu bytes, need %zu for N=%lld", fn, ws_bytes, L.total,
              (long long)N);
    return SUBM3D_ERR_WORKSPACE;
  }
  int* err = nullptr;
  if (!sync) {
    err = forward_error_word();
    if (!err) return SUBM3D_ERR_CUDA;
  }
  char* ws = static_cast<char*>(workspace);
  KmapStatus* st = reinterpret_cast<KmapStatus*>(ws + L.status);
  unsigned long long* mk0 = reinterpret_cast<unsigned long long*>(ws + L.mk0);
  unsigned long long* mk1 = reinterpret_cast<unsigned long long*>(ws + L.mk1);
  int32_t* ix0 = reinterpret_cast<int32_t*>(ws + L.ix0);
  int32_t* ix1 = reinterpret_cast<int32_t*>(ws + L.ix1);
  Slot* table = reinterpret_cast<Slot*>(ws + L.table);
  int bits = 2;   // bits per axis of the sort key (as launch_sort chooses them)
  while ((1 << bits) < res) ++bits;

  const int4* c4 = reinterpret_cast<const int4*>(coords);
  // the hashed front end (slot indices are kept as 32-bit words, so only while the
  // full-size table has at most 2^31 slots); the radix sort of all voxels otherwise, and
  // to name the first repeated row of a build that found a duplicate
  const bool hashed = !force_sorted && cap_max <= (int64_t(1) << 31);
  g_stage.begin(stream);
  if (hashed) {
    int64_t cap0 = hash_capacity;
    if (cap0 == 0) {
      cap0 = 64;
      while (cap0 < N / 4 && cap0 < cap_max) cap0 <<= 1;
    }
    const bool can_grow = hash_capacity == 0 && cap0 < cap_max;
    uint32_t* slot_of = reinterpret_cast<uint32_t*>(ix1);   // per voxel, input order
    int32_t* bv1 = reinterpret_cast<int32_t*>(ws + L.bv1);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
    uint32_t* hist2 = L.hist2 ? reinterpret_cast<uint32_t*>(ws + L.hist2) : nullptr;
    kmap_h_init<<<grid_for(cap0, 256, 8), 256, 0, stream>>>(table, cap0, hist, hist2, st);
    SUBM3D_LAUNCHED("kmap_h_init");
    kmap_h_insert<<<grid_for(N, 256, 8), 256, 0, stream>>>(c4, N, res, bits, table, slot_of,
                                                           false, can_grow, st);
    SUBM3D_LAUNCHED("kmap_h_insert");
    if (can_grow) {   // both return at once unless the first table was too small
      kmap_h_grow<<<grid_for(cap_max, 256, 8), 256, 0, stream>>>(table, cap_max, st);
      SUBM3D_LAUNCHED("kmap_h_grow");
      kmap_h_insert<<<grid_for(N, 256, 8), 256, 0, stream>>>(c4, N, res, bits, table, slot_of,
                                                             true, false, st);
      SUBM3D_LAUNCHED("kmap_h_insert");
    }
    g_stage.mark("block insert", stream);
    // the occupied blocks (key, slot) into (mk0, ix0), sorted by key through (mk1, bv1)
    kmap_h_compact<<<grid_for(cap0, 256, 8), 256, 0, stream>>>(table, mk0, ix0, st);
    SUBM3D_LAUNCHED("kmap_h_compact");
    const int npass_b = (3 * bits - 6 + 16 + 7) / 8;
    kmap_plan<<<1, 1, 0, stream>>>(npass_b, -1, st);
    SUBM3D_LAUNCHED("kmap_plan");
    g_stage.mark("block compact", stream);
    const int* plans = reinterpret_cast<const int*>(reinterpret_cast<const char*>(st) +
                                                    offsetof(KmapStatus, plan));
    const int rc = launch_radix(mk0, mk1, ix0, bv1, N, npass_b, hist, ws + L.cnt, L.nblk, plans,
                                st, stream, "block sort pass", &st->nblocks, true);
    if (rc != SUBM3D_OK) return rc;
    // the scan's published counts reuse the sort's status words (cleared by its
    // histogram kernel, then tagged by its passes, never with the scan's tag)
    unsigned long long* scan_status = sort_scratch(ws + L.cnt, L.nblk).status;
    kmap_h_starts<<<grid_for((N + kStartTile - 1) / kStartTile * 256, 256, 4), 256, 0, stream>>>(
        ix0, bv1, table, scan_status, N, st);
    SUBM3D_LAUNCHED("kmap_h_starts");
    g_stage.mark("block starts", stream);
    kmap_h_scatter<<<grid_for(N, 256, 8), 256, 0, stream>>>(c4, slot_of, N, bits, table, mk0, ix0,
                                                            order, st);
    SUBM3D_LAUNCHED("kmap_h_scatter");
    g_stage.mark("voxel scatter", stream);
  } else {
    const int rc = launch_sort(c4, N, res, L, ws, stream);
    if (rc != SUBM3D_OK) return rc;
    kmap_blocks_count<<<grid_for(N, 256, 4), 256, 0, stream>>>(mk0, mk1, ix0, ix1, N, order, st);
    SUBM3D_LAUNCHED("kmap_blocks_count");
    kmap_table_init<<<grid_for(cap_max, 256, 8), 256, 0, stream>>>(table, hash_capacity, cap_max,
                                                                  st);
    SUBM3D_LAUNCHED("kmap_table_init");
    kmap_blocks_insert<<<grid_for(N, 256, 8), 256, 0, stream>>>(c4, mk0, mk1, ix0, ix1, N, table,
                                                                st);
    SUBM3D_LAUNCHED("kmap_blocks_insert");
    g_stage.mark("block table", stream);
  }
  // the probe's grid is exactly the blocks that fit on the GPU at once (its shared memory
  // limits them), so that its grid-stride loop runs in one wave
  static PerDevice<int> probe_fit[2];
  int fit = 0;
  {
    const int mode = grouped ? 1 : 0;
    const int rc = probe_fit[mode].get(&fit, [mode](int* v) -> int {
      int n = 0;
      const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, mode ? reinterpret_cast<const void*>(kmap_probe<kProbeSorted>)
                   : reinterpret_cast<const void*>(kmap_probe<kProbeNbr>),
          kProbeThreads, 0);
      *v = (e == cudaSuccess && n > 0) ? n : 4;
      return static_cast<int>(SUBM3D_OK);
    });
    if (rc != SUBM3D_OK) return rc;
  }
  const int probe_grid = grid_for((N + 31) / 32 * 32, kProbeThreads, fit);
  if (!grouped) {
    kmap_probe<kProbeNbr><<<probe_grid, kProbeThreads, 0, stream>>>(
        mk0, mk1, ix0, ix1, N, res, bits, table, nbr, nullptr, nullptr, 0, nullptr, nullptr, st);
    SUBM3D_LAUNCHED("kmap_probe");
    g_stage.mark("probe", stream);
  } else {
    char* pl = static_cast<char*>(plan);
    int32_t* perm = reinterpret_cast<int32_t*>(pl + PL.perm);
    int32_t* pnbr = reinterpret_cast<int32_t*>(pl + PL.nbr);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(pl + PL.tmask);
    unsigned long long* k2a = reinterpret_cast<unsigned long long*>(ws + L.k2a);
    unsigned long long* k2b = reinterpret_cast<unsigned long long*>(ws + L.k2b);
    int32_t* v2a = reinterpret_cast<int32_t*>(ws + L.v2a);
    int32_t* v2b = reinterpret_cast<int32_t*>(ws + L.v2b);
    int32_t* nbr_sorted = reinterpret_cast<int32_t*>(ws + L.nbr_sorted);
    uint32_t* hist2 = reinterpret_cast<uint32_t*>(ws + L.hist2);
    int wshift = 0;
    while ((int64_t(1) << wshift) < window) ++wshift;
    const int64_t last_window = (N - 1) >> wshift;
    int wbits = 0;
    while ((last_window >> wbits) != 0) ++wbits;
    const int npass2 = (27 + wbits + 7) / 8;
    if (window == 1) {
      // Windows of one voxel: the stable sort by (position, mask) is the identity, so the
      // plan is the Morton order itself: the probe writes its rows straight into the
      // plan, with perm, and ORs each warp's masks into its tile's (cleared first; the
      // four warps of a probe block hold one 128-row tile).
      SUBM3D_CUDA_TRY(cudaMemsetAsync(tmask, 0, sizeof(uint32_t) * PL.ntiles, stream));
      kmap_probe<kProbeSorted><<<probe_grid, kProbeThreads, 0, stream>>>(
          mk0, mk1, ix0, ix1, N, res, bits, table, pnbr, nullptr, nullptr, 0, perm, tmask, st);
      SUBM3D_LAUNCHED("kmap_probe_sorted");
      g_stage.mark("probe (Morton order) + plan", stream);
    } else {
      kmap_probe<kProbeSorted><<<probe_grid, kProbeThreads, 0, stream>>>(
          mk0, mk1, ix0, ix1, N, res, bits, table, nbr_sorted, k2a, v2a, wshift, nullptr, nullptr,
          st);
      SUBM3D_LAUNCHED("kmap_probe_sorted");
      g_stage.mark("probe (Morton order) + masks", stream);
      kmap_plan2<<<1, 1, 0, stream>>>(npass2, st);
      SUBM3D_LAUNCHED("kmap_plan2");
      const int* plans2 = reinterpret_cast<const int*>(reinterpret_cast<const char*>(st) +
                                                       offsetof(KmapStatus, plan2));
      const int rc = launch_radix(k2a, k2b, v2a, v2b, N, npass2, hist2, ws + L.cnt, L.nblk,
                                  plans2, st, stream, "grouping sort pass");
      if (rc != SUBM3D_OK) return rc;
      kmap_plan_index<<<grid_for(PL.ntiles * 128, 128, 16), 128, 0, stream>>>(
          k2a, k2b, v2a, v2b, ix0, ix1, N, PL.ntiles, nbr_sorted, perm, pnbr, tmask, st);
      SUBM3D_LAUNCHED("kmap_plan_index");
      g_stage.mark("plan index + rows", stream);
    }
  }

  if (!sync) {
    kmap_report<<<1, 1, 0, stream>>>(st, err);
    SUBM3D_LAUNCHED("kmap_report");
    return SUBM3D_OK;
  }
  KmapStatus host;
  SUBM3D_CUDA_TRY(cudaMemcpyAsync(&host, st, sizeof(host), cudaMemcpyDeviceToHost, stream));
  SUBM3D_CUDA_TRY(cudaStreamSynchronize(stream));
  if (host.flags & kFlagCoord) {
    set_error("%s: coordinate row %lld outside 0<=b<=%d, 0<=z,y,x<%d", fn, host.bad_row,
              SUBM3D_MAX_BATCH, res);
    return SUBM3D_ERR_COORD_RANGE;
  }
  if (hashed && (host.flags & kFlagDup)) {
    // the hashed front end knows that two rows share a coordinate, not which row is the
    // first repeat (that depends on the order of its atomics): the sorted build says so
    return kmap_run(fn, coords, N, res, nbr, order, hash_capacity, window, plan, plan_bytes,
                    workspace, ws_bytes, sync, stream, true);
  }
  if (host.flags & kFlagInternal) {
    set_error("%s: internal error (sort or block table produced an index outside [0, N))", fn);
    return SUBM3D_ERR_DEVICE;
  }
  if (host.flags & kFlagDup) {
    set_error("%s: duplicate coordinate (row %lld repeats an earlier row)", fn, host.bad_row);
    return SUBM3D_ERR_DUPLICATE;
  }
  if (host.flags & kFlagFull) {
    set_error("%s: %llu occupied 4x4x4 blocks do not fit a hash capacity of %llu within %d "
              "probes (N=%lld)",
              fn, host.nblocks, host.cap, kMaxProbe, (long long)N);
    return SUBM3D_ERR_HASH_FULL;
  }
  return SUBM3D_OK;
}

}  // namespace

void kmap_stage_timing(bool on) {
  // the events are made here, not during a build (making one takes far longer than a
  // small stage runs)
  if (on)
    for (int i = 0; i < StageTimer::kMax; ++i)
      if (!g_stage.ev[i] && cudaEventCreate(&g_stage.ev[i]) != cudaSuccess) break;
  g_stage.on = on;
}

int kmap_stage_times(float* ms, const char** names, int max) {
  const int n = g_stage.n;
  if (n < 2) return 0;
  SUBM3D_CUDA_TRY(cudaEventSynchronize(g_stage.ev[n - 1]));
  int k = 0;
  for (int i = 1; i < n && k < max; ++i, ++k) {
    SUBM3D_CUDA_TRY(cudaEventElapsedTime(&ms[k], g_stage.ev[i - 1], g_stage.ev[i]));
    names[k] = g_stage.name[i];
  }
  return k;
}

int kmap_build(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr, int32_t* order,
               int64_t hash_capacity, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return kmap_run("subm3d_build_kmap", coords, N, res, nbr, order, hash_capacity, 0, nullptr, 0,
                  workspace, ws_bytes, true, stream);
}

int kmap_build_async(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                     void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return kmap_run("subm3d_build_kmap_async", coords, N, res, nbr, nullptr, 0, 0, nullptr, 0,
                  workspace, ws_bytes, false, stream);
}

size_t kmap_grouped_workspace_bytes(int64_t N) {
  if (N < 0 || N > 0x7FFFFFFFll) return 0;
  return make_layout(N, default_hash_capacity(N), true).total;
}

int kmap_build_grouped(const int32_t* coords, int64_t N, int32_t res, int64_t window, void* plan,
                       size_t plan_bytes, void* workspace, size_t ws_bytes, bool sync,
                       cudaStream_t stream) {
  if (!plan && N > 0) {
    set_error("subm3d_build_kmap_grouped: plan is NULL");
    return SUBM3D_ERR_ARG;
  }
  return kmap_run("subm3d_build_kmap_grouped", coords, N, res, nullptr, nullptr, 0,
                  window ? window : SUBM3D_GROUP_WINDOW, plan, plan_bytes,
                  workspace, ws_bytes, sync, stream);
}

size_t downsample_workspace_bytes(int64_t N) {
  if (N < 0 || N > 0x7FFFFFFFll) return 0;
  return make_ds_layout(N).total;
}

namespace {
template <typename T>
int launch_pool(const void* feats, int C, const int32_t* ix0, const int32_t* ix1,
                const int32_t* pstart, const uint32_t* m_dev, int64_t M_max, int mode, void* out,
                const KmapStatus* st, cudaStream_t stream) {
  constexpr int V = 16 / sizeof(T);
  const T* f = static_cast<const T*>(feats);
  T* o = static_cast<T*>(out);
  if (C % V == 0) {
    ds_pool<T, V><<<grid_for(M_max * (C / V), 256, 8), 256, 0, stream>>>(f, C, ix0, ix1, pstart,
                                                                         m_dev, mode, o, st);
  } else {
    ds_pool<T, 1><<<grid_for(M_max * C, 256, 8), 256, 0, stream>>>(f, C, ix0, ix1, pstart, m_dev,
                                                                   mode, o, st);
  }
  SUBM3D_LAUNCHED("ds_pool");
  return SUBM3D_OK;
}
template <typename T>
int launch_unpool(const void* coarse, int64_t M, int C, const int32_t* parent, int64_t N,
                  void* fine, cudaStream_t stream) {
  constexpr int V = 16 / sizeof(T);
  const T* c = static_cast<const T*>(coarse);
  T* f = static_cast<T*>(fine);
  int* err = forward_error_word();
  if (!err) return SUBM3D_ERR_CUDA;
  if (C % V == 0) {
    us_gather<T, V><<<grid_for(N * (C / V), 256, 8), 256, 0, stream>>>(c, M, C, parent, N, f, err);
  } else {
    us_gather<T, 1><<<grid_for(N * C, 256, 8), 256, 0, stream>>>(c, M, C, parent, N, f, err);
  }
  SUBM3D_LAUNCHED("us_gather");
  return SUBM3D_OK;
}
}  // namespace

// Asynchronous downsample: M (0 after an error) into the caller's device word, the
// status folded into the device error word.
__global__ void ds_report(const KmapStatus* st, int64_t N, int64_t* M_dev, int* err) {
  const int f = st->flags;
  int bits = 0;
  if (f & kFlagOrder) bits |= kDevErrBadOrder;
  if (f & kFlagCoord) bits |= kDevErrKmapCoord;
  if (f & kFlagDup) bits |= kDevErrKmapDup;
  if (f & kFlagInternal) bits |= kDevErrKmapInternal;
  const long long M = static_cast<long long>(st->nblocks);
  if (!bits && (M < 1 || M > N)) bits |= kDevErrKmapInternal;
  *M_dev = bits ? 0 : M;
  if (bits) atomicOr(err, bits);
}

int downsample_build(const int32_t* coords, int64_t N, int32_t res, const int32_t* order,
                     const void* feats, int32_t C, subm3d_dtype dtype, int mode,
                     int32_t* coarse_coords, void* coarse_feats, int32_t* parent,
                     uint8_t* child_mask, int64_t* M_out, void* workspace, size_t ws_bytes,
                     cudaStream_t stream, int64_t* M_dev) {
  if (!M_out && !M_dev) {
    set_error("subm3d_downsample: M_out (host) is NULL");
    return SUBM3D_ERR_ARG;
  }
  if (M_out) *M_out = 0;
  if (M_dev && (reinterpret_cast<uintptr_t>(M_dev) & 7)) {
    set_error("subm3d_downsample_async: M=%p must be 8-byte aligned", (void*)M_dev);
    return SUBM3D_ERR_ARG;
  }
  if (N < 0 || N > 0x7FFFFFFFll) {
    set_error("subm3d_downsample: N=%lld outside [0, 2^31)", (long long)N);
    return SUBM3D_ERR_ARG;
  }
  if (res < 1 || res > SUBM3D_MAX_RES) {
    set_error("subm3d_downsample: res=%d outside [1, %d]", res, SUBM3D_MAX_RES);
    return SUBM3D_ERR_ARG;
  }
  if (mode != SUBM3D_POOL_MEAN && mode != SUBM3D_POOL_MAX) {
    set_error("subm3d_downsample: unknown pooling mode %d", mode);
    return SUBM3D_ERR_ARG;
  }
  if (feats && (C < 1 || C > 4096 || (dtype != SUBM3D_F32 && dtype != SUBM3D_BF16))) {
    set_error("subm3d_downsample: C=%d must lie in [1, 4096] and dtype %d be F32 or BF16", C,
              static_cast<int>(dtype));
    return SUBM3D_ERR_ARG;
  }
  if (N == 0) {
    if (M_dev) SUBM3D_CUDA_TRY(cudaMemsetAsync(M_dev, 0, sizeof(int64_t), stream));
    return SUBM3D_OK;
  }
  if (!coords || !coarse_coords || !parent || !child_mask || !workspace || (feats && !coarse_feats)) {
    set_error("subm3d_downsample: NULL pointer (coords=%p coarse_coords=%p parent=%p "
              "child_mask=%p workspace=%p feats=%p coarse_feats=%p)",
              (const void*)coords, (void*)coarse_coords, (void*)parent, (void*)child_mask,
              workspace, feats, coarse_feats);
    return SUBM3D_ERR_ARG;
  }
  const uintptr_t any = reinterpret_cast<uintptr_t>(coords) |
                        reinterpret_cast<uintptr_t>(coarse_coords) |
                        reinterpret_cast<uintptr_t>(parent) | reinterpret_cast<uintptr_t>(feats) |
                        reinterpret_cast<uintptr_t>(coarse_feats);
  if (any & 15) {
    set_error("subm3d_downsample: coords, coarse_coords, parent, feats and coarse_feats must be "
              "16-byte aligned");
    return SUBM3D_ERR_ARG;
  }
  const DsLayout D = make_ds_layout(N);
  if (reinterpret_cast<uintptr_t>(workspace) & 255) {
    set_error("subm3d_downsample: workspace=%p must be 256-byte aligned", workspace);
    return SUBM3D_ERR_WORKSPACE;
  }
  if (ws_bytes < D.total) {
    set_error("subm3d_downsample: workspace of %zu bytes, need %zu for N=%lld", ws_bytes, D.total,
              (long long)N);
    return SUBM3D_ERR_WORKSPACE;
  }
  char* ws = static_cast<char*>(workspace);
  const Layout& L = D.k;
  KmapStatus* st = reinterpret_cast<KmapStatus*>(ws + L.status);
  unsigned long long* mk0 = reinterpret_cast<unsigned long long*>(ws + L.mk0);
  unsigned long long* mk1 = reinterpret_cast<unsigned long long*>(ws + L.mk1);
  int32_t* ix0 = reinterpret_cast<int32_t*>(ws + L.ix0);
  int32_t* ix1 = reinterpret_cast<int32_t*>(ws + L.ix1);
  uint32_t* tsum = reinterpret_cast<uint32_t*>(ws + D.tsum);
  int32_t* pstart = reinterpret_cast<int32_t*>(ws + D.pstart);
  const int4* c4 = reinterpret_cast<const int4*>(coords);
  if (order) {   // the caller's Morton order: keys gathered in that order, no sort
    if (reinterpret_cast<uintptr_t>(order) & 15) {
      set_error("subm3d_downsample_sorted: order=%p must be 16-byte aligned", (const void*)order);
      return SUBM3D_ERR_ARG;
    }
    int bits = 2;
    while ((1 << bits) < res) ++bits;
    kmap_init<<<8, 256, 0, stream>>>(st, reinterpret_cast<uint32_t*>(ws + L.hist), nullptr);
    SUBM3D_LAUNCHED("kmap_init");
    ds_keys_in_order<<<grid_for(N, 256, 8), 256, 0, stream>>>(c4, order, N, res, bits, mk0, ix0, st);
    SUBM3D_LAUNCHED("ds_keys_in_order");
  } else {
    const int rc = launch_sort(c4, N, res, L, ws, stream);
    if (rc != SUBM3D_OK) return rc;
  }
  const int ntile = static_cast<int>(D.ntile);
  ds_count<<<ntile, kSortThreads, 0, stream>>>(mk0, mk1, ix0, ix1, N, tsum, st);
  SUBM3D_LAUNCHED("ds_count");
  ds_scan<<<1, 256, 0, stream>>>(tsum, D.ntile, st);
  SUBM3D_LAUNCHED("ds_scan");
  int bits = 2;
  while ((1 << bits) < res) ++bits;
  ds_emit<<<ntile, kSortThreads, 0, stream>>>(c4, mk0, mk1, ix0, ix1, N, tsum,
                                              reinterpret_cast<int4*>(coarse_coords), parent,
                                              child_mask, pstart, bits, st);
  SUBM3D_LAUNCHED("ds_emit");
  if (feats) {   // enqueued before the wait: M is read on the device
    const int prc =
        dtype == SUBM3D_BF16
            ? launch_pool<__nv_bfloat16>(feats, C, ix0, ix1, pstart, tsum + D.ntile, N, mode,
                                         coarse_feats, st, stream)
            : launch_pool<float>(feats, C, ix0, ix1, pstart, tsum + D.ntile, N, mode,
                                 coarse_feats, st, stream);
    if (prc != SUBM3D_OK) return prc;
  }
  if (M_dev) {   // no wait: M and the status stay on the device
    int* err = forward_error_word();
    if (!err) return SUBM3D_ERR_CUDA;
    ds_report<<<1, 1, 0, stream>>>(st, N, M_dev, err);
    SUBM3D_LAUNCHED("ds_report");
    return SUBM3D_OK;
  }

  KmapStatus host;
  SUBM3D_CUDA_TRY(cudaMemcpyAsync(&host, st, sizeof(host), cudaMemcpyDeviceToHost, stream));
  SUBM3D_CUDA_TRY(cudaStreamSynchronize(stream));
  if (host.flags & kFlagOrder) {
    set_error("subm3d_downsample_sorted: order[%lld] does not continue the Morton order of the "
              "coordinates (a row outside [0, N), a coordinate outside the grid, or a smaller key)",
              host.bad_row);
    return SUBM3D_ERR_ARG;
  }
  if (host.flags & kFlagCoord) {
    set_error("subm3d_downsample: coordinate row %lld outside 0<=b<=%d, 0<=z,y,x<%d",
              host.bad_row, SUBM3D_MAX_BATCH, res);
    return SUBM3D_ERR_COORD_RANGE;
  }
  if (host.flags & kFlagInternal) {
    set_error("subm3d_downsample: internal error (the sort produced an index outside [0, N))");
    return SUBM3D_ERR_DEVICE;
  }
  if (host.flags & kFlagDup) {
    set_error("subm3d_downsample: duplicate coordinate (row %lld repeats an earlier row)",
              host.bad_row);
    return SUBM3D_ERR_DUPLICATE;
  }
  const int64_t M = static_cast<int64_t>(host.nblocks);
  if (M < 1 || M > N) {
    set_error("subm3d_downsample: internal error (%lld parents for %lld voxels)", (long long)M,
              (long long)N);
    return SUBM3D_ERR_DEVICE;
  }
  *M_out = M;
  return SUBM3D_OK;
}

int upsample_launch(const void* coarse_feats, int64_t M, int32_t C, const int32_t* parent,
                    int64_t N, subm3d_dtype dtype, void* fine_feats, cudaStream_t stream) {
  if (N < 0 || N > 0x7FFFFFFFll || M < 0 || M > 0x7FFFFFFFll) {
    set_error("subm3d_upsample: N=%lld, M=%lld outside [0, 2^31)", (long long)N, (long long)M);
    return SUBM3D_ERR_ARG;
  }
  if (C < 1 || C > 4096 || (dtype != SUBM3D_F32 && dtype != SUBM3D_BF16)) {
    set_error("subm3d_upsample: C=%d must lie in [1, 4096] and dtype %d be F32 or BF16", C,
              static_cast<int>(dtype));
    return SUBM3D_ERR_ARG;
  }
  if (N == 0) return SUBM3D_OK;
  if (!parent || !fine_feats || (M > 0 && !coarse_feats)) {
    set_error("subm3d_upsample: NULL pointer (coarse_feats=%p parent=%p fine_feats=%p)",
              coarse_feats, (const void*)parent, fine_feats);
    return SUBM3D_ERR_ARG;
  }
  const uintptr_t any = reinterpret_cast<uintptr_t>(coarse_feats) |
                        reinterpret_cast<uintptr_t>(parent) | reinterpret_cast<uintptr_t>(fine_feats);
  if (any & 15) {
    set_error("subm3d_upsample: coarse_feats=%p parent=%p fine_feats=%p must be 16-byte aligned",
              coarse_feats, (const void*)parent, fine_feats);
    return SUBM3D_ERR_ARG;
  }
  return dtype == SUBM3D_BF16
             ? launch_unpool<__nv_bfloat16>(coarse_feats, M, C, parent, N, fine_feats, stream)
             : launch_unpool<float>(coarse_feats, M, C, parent, N, fine_feats, stream);
}

namespace {
template <typename T>
int launch_s2c(const void* feats, const int4* coords, const int32_t* parent,
               const uint8_t* mask, int64_t N, int64_t M, int C, void* out, cudaStream_t stream) {
  constexpr int V = 16 / sizeof(T);
  const T* f = static_cast<const T*>(feats);
  T* o = static_cast<T*>(out);
  const bool vec = C % V == 0;
  int* err = N > 0 ? forward_error_word() : nullptr;
  if (N > 0 && !err) return SUBM3D_ERR_CUDA;
  if (M > 0) {
    if (vec) {
      s2c_zero<T, V><<<grid_for(M * 8 * (C / V), 256, 8), 256, 0, stream>>>(mask, M, C, o);
    } else {
      s2c_zero<T, 1><<<grid_for(M * 8 * C, 256, 8), 256, 0, stream>>>(mask, M, C, o);
    }
    SUBM3D_LAUNCHED("s2c_zero");
  }
  if (N > 0) {
    if (vec) {
      s2c_scatter<T, V><<<grid_for(N * (C / V), 256, 8), 256, 0, stream>>>(
          f, coords, parent, N, M, C, o, err);
    } else {
      s2c_scatter<T, 1><<<grid_for(N * C, 256, 8), 256, 0, stream>>>(f, coords, parent, N, M, C,
                                                                    o, err);
    }
    SUBM3D_LAUNCHED("s2c_scatter");
  }
  return SUBM3D_OK;
}
template <typename T>
int launch_c2s(const void* coarse, const int4* coords, const int32_t* parent, int64_t N, int64_t M,
               int C, void* fine, cudaStream_t stream) {
  constexpr int V = 16 / sizeof(T);
  const T* c = static_cast<const T*>(coarse);
  T* f = static_cast<T*>(fine);
  int* err = forward_error_word();
  if (!err) return SUBM3D_ERR_CUDA;
  if (C % V == 0) {
    c2s_gather<T, V><<<grid_for(N * (C / V), 256, 8), 256, 0, stream>>>(c, coords, parent, N, M,
                                                                         C, f, err);
  } else {
    c2s_gather<T, 1><<<grid_for(N * C, 256, 8), 256, 0, stream>>>(c, coords, parent, N, M, C, f,
                                                                 err);
  }
  SUBM3D_LAUNCHED("c2s_gather");
  return SUBM3D_OK;
}

int check_pixel_args(const char* fn, int64_t N, int64_t M, int32_t C, subm3d_dtype dtype) {
  if (N < 0 || N > 0x7FFFFFFFll || M < 0 || M > 0x7FFFFFFFll) {
    set_error("%s: N=%lld, M=%lld outside [0, 2^31)", fn, (long long)N, (long long)M);
    return SUBM3D_ERR_ARG;
  }
  if (C < 1 || C > 4096 || (dtype != SUBM3D_F32 && dtype != SUBM3D_BF16)) {
    set_error("%s: C=%d must lie in [1, 4096] and dtype %d be F32 or BF16", fn, C,
              static_cast<int>(dtype));
    return SUBM3D_ERR_ARG;
  }
  return SUBM3D_OK;
}
}  // namespace

int spatial2channel_launch(const void* feats, const int32_t* coords, const int32_t* parent,
                           const uint8_t* child_mask, int64_t N, int64_t M, int32_t C,
                           subm3d_dtype dtype, void* out, cudaStream_t stream) {
  const int rc = check_pixel_args("subm3d_spatial2channel", N, M, C, dtype);
  if (rc != SUBM3D_OK) return rc;
  if ((N > 0 && (!feats || !coords || !parent)) || (M > 0 && (!child_mask || !out))) {
    set_error("subm3d_spatial2channel: NULL pointer (feats=%p coords=%p parent=%p child_mask=%p "
              "out=%p)",
              feats, (const void*)coords, (const void*)parent, (const void*)child_mask, out);
    return SUBM3D_ERR_ARG;
  }
  const uintptr_t any = reinterpret_cast<uintptr_t>(feats) | reinterpret_cast<uintptr_t>(coords) |
                        reinterpret_cast<uintptr_t>(parent) | reinterpret_cast<uintptr_t>(out);
  if (any & 15) {
    set_error("subm3d_spatial2channel: feats, coords, parent and out must be 16-byte aligned");
    return SUBM3D_ERR_ARG;
  }
  const int4* c4 = reinterpret_cast<const int4*>(coords);
  return dtype == SUBM3D_BF16
             ? launch_s2c<__nv_bfloat16>(feats, c4, parent, child_mask, N, M, C, out, stream)
             : launch_s2c<float>(feats, c4, parent, child_mask, N, M, C, out, stream);
}

int channel2spatial_launch(const void* coarse_feats, const int32_t* coords, const int32_t* parent,
                           int64_t N, int64_t M, int32_t C, subm3d_dtype dtype, void* fine_feats,
                           cudaStream_t stream) {
  const int rc = check_pixel_args("subm3d_channel2spatial", N, M, C, dtype);
  if (rc != SUBM3D_OK) return rc;
  if (N == 0) return SUBM3D_OK;
  if (!coords || !parent || !fine_feats || (M > 0 && !coarse_feats)) {
    set_error("subm3d_channel2spatial: NULL pointer (coarse_feats=%p coords=%p parent=%p "
              "fine_feats=%p)",
              coarse_feats, (const void*)coords, (const void*)parent, fine_feats);
    return SUBM3D_ERR_ARG;
  }
  const uintptr_t any = reinterpret_cast<uintptr_t>(coarse_feats) |
                        reinterpret_cast<uintptr_t>(coords) | reinterpret_cast<uintptr_t>(parent) |
                        reinterpret_cast<uintptr_t>(fine_feats);
  if (any & 15) {
    set_error("subm3d_channel2spatial: coarse_feats, coords, parent and fine_feats must be "
              "16-byte aligned");
    return SUBM3D_ERR_ARG;
  }
  const int4* c4 = reinterpret_cast<const int4*>(coords);
  return dtype == SUBM3D_BF16
             ? launch_c2s<__nv_bfloat16>(coarse_feats, c4, parent, N, M, C, fine_feats, stream)
             : launch_c2s<float>(coarse_feats, c4, parent, N, M, C, fine_feats, stream);
}

}  // namespace subm3d
