// Kernel-map build for submanifold convolution: for every active voxel, the input
// index of each of its 27 neighbours (-1 when absent).
//
// The submanifold variant (outputs only at active sites; "pixal3d_mrp_mlx
// CLAUDE.md", "Measured facts": stride 1 / no padding dispatches to SubMConv3d)
// needs exactly this table; the pages' "spatial cache" (README scope table) is what
// lets one table serve several convolutions on one voxel set.
//
// Pipeline (one stream, one host sync at the end to read the status word):
//   1. init    : status word, digit histograms and hash table cleared
//   2. pack    : validate (b, z, y, x), packed key b<<48|z<<32|y<<16|x, sort key
//                (b << 3*bits) | Morton(z, y, x), all-pass digit histograms
//   3. plan    : which 8-bit radix passes are not constant (others are skipped)
//   4. passes  : LSD radix sort of (sort key, row) -- count / scan / stable scatter
//   5. insert  : keys into an open-addressing table in Morton order (atomicCAS,
//                bounded linear probing; equal keys = duplicate coordinates)
//   6. probe   : a warp takes 32 consecutive voxels and spreads their 32 x 27
//                (voxel, offset) lookups over its lanes, so lane l of round t
//                writes nbr[v0*27 + 32 t + l]: fully coalesced rows of the table.
//
// Hash: a slot is 16 bytes {key, row}; the home slot of a key is
// mix(key of its 2x2x2 block) * 8 + (position inside the block), so the 27
// lookups of a voxel touch at most eight 128-byte lines and neighbouring voxels
// share them. mix is the splitmix64 finaliser (Steele, Lea and Flood, 2014).
#include "common.cuh"

namespace subm3d {
namespace {

constexpr unsigned long long kEmptyKey = ~0ull;
constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;   // keys per sort block
constexpr int kMaxPasses = 8;
constexpr int kMaxProbe = 4096;

enum : int { kFlagCoord = 1, kFlagDup = 2, kFlagFull = 4, kFlagInternal = 8 };

struct KmapStatus {
  int flags;
  int pad;
  long long bad_row;
  int plan[kMaxPasses + 1];   // plan[p]: bit1 = pass active, bit0 = source buffer; plan[8] = final buffer
};

struct __align__(16) Slot {
  unsigned long long key;
  int row;
  int pad;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t status, hist, keys, mk0, mk1, ix0, ix1, cnt, table, total;
  int64_t nblk;
};

Layout make_layout(int64_t N, int64_t cap) {
  Layout L;
  L.nblk = (N + kSortTile - 1) / kSortTile;
  size_t o = 0;
  L.status = o; o = align256(o + sizeof(KmapStatus));
  L.hist = o;   o = align256(o + sizeof(uint32_t) * kMaxPasses * 256);
  L.keys = o;   o = align256(o + sizeof(uint64_t) * N);
  L.mk0 = o;    o = align256(o + sizeof(uint64_t) * N);
  L.mk1 = o;    o = align256(o + sizeof(uint64_t) * N);
  L.ix0 = o;    o = align256(o + sizeof(int32_t) * N);
  L.ix1 = o;    o = align256(o + sizeof(int32_t) * N);
  L.cnt = o;    o = align256(o + sizeof(uint32_t) * 256 * L.nblk);
  L.table = o;  o = align256(o + sizeof(Slot) * cap);
  L.total = o;
  return L;
}

__device__ __forceinline__ unsigned long long pack_key(int b, int z, int y, int x) {
  return (static_cast<unsigned long long>(static_cast<uint32_t>(b) & 0xFFFFu) << 48) |
         (static_cast<unsigned long long>(static_cast<uint32_t>(z) & 0xFFFFu) << 32) |
         (static_cast<unsigned long long>(static_cast<uint32_t>(y) & 0xFFFFu) << 16) |
         static_cast<unsigned long long>(static_cast<uint32_t>(x) & 0xFFFFu);
}

// Interleaves the low `bits` bits of z, y, x: bit t of x -> 3t, of y -> 3t+1, of z -> 3t+2.
__device__ __forceinline__ unsigned long long morton3(uint32_t z, uint32_t y, uint32_t x, int bits) {
  unsigned long long m = 0;
  for (int t = 0; t < bits; ++t) {
    m |= static_cast<unsigned long long>((x >> t) & 1u) << (3 * t);
    m |= static_cast<unsigned long long>((y >> t) & 1u) << (3 * t + 1);
    m |= static_cast<unsigned long long>((z >> t) & 1u) << (3 * t + 2);
  }
  return m;
}

__device__ __forceinline__ unsigned long long mix64(unsigned long long v) {
  v = (v ^ (v >> 30)) * 0xbf58476d1ce4e5b9ull;
  v = (v ^ (v >> 27)) * 0x94d049bb133111ebull;
  return v ^ (v >> 31);
}

__device__ __forceinline__ unsigned long long home_slot(unsigned long long key,
                                                        unsigned long long mask) {
  const unsigned long long low = 0x0000000100010001ull;   // lowest bit of z, y and x
  const unsigned long long inner = ((key >> 30) & 4ull) | ((key >> 15) & 2ull) | (key & 1ull);
  return ((mix64(key & ~low) << 3) | inner) & mask;
}

// 1. ------------------------------------------------------------------------------
__global__ void kmap_init(KmapStatus* st, uint32_t* hist, Slot* table, int64_t cap) {
  const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  if (tid == 0) {
    st->flags = 0;
    st->pad = 0;
    st->bad_row = 0x7FFFFFFFFFFFFFFFll;
    for (int p = 0; p <= kMaxPasses; ++p) st->plan[p] = 0;
  }
  for (int64_t i = tid; i < kMaxPasses * 256; i += stride) hist[i] = 0;
  for (int64_t i = tid; i < cap; i += stride) {
    Slot s;
    s.key = kEmptyKey;
    s.row = -1;
    s.pad = 0;
    table[i] = s;
  }
}

// 2. ------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) kmap_pack(const int4* __restrict__ coords, int64_t N,
                                                 int res, int bits, int npass,
                                                 unsigned long long* __restrict__ keys,
                                                 unsigned long long* __restrict__ mk,
                                                 int32_t* __restrict__ ix, uint32_t* hist,
                                                 KmapStatus* st) {
  __shared__ uint32_t sh[kMaxPasses][256];
  for (int i = threadIdx.x; i < kMaxPasses * 256; i += blockDim.x) (&sh[0][0])[i] = 0;
  __syncthreads();
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
    const unsigned long long key = pack_key(c.x, c.y, c.z, c.w);
    const unsigned long long m =
        (static_cast<unsigned long long>(c.x) << (3 * bits)) | morton3(c.y, c.z, c.w, bits);
    keys[i] = key;
    mk[i] = m;
    ix[i] = static_cast<int32_t>(i);
    for (int p = 0; p < npass; ++p) atomicAdd(&sh[p][(m >> (8 * p)) & 255u], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < npass * 256; i += blockDim.x) {
    const uint32_t v = (&sh[0][0])[i];
    if (v) atomicAdd(&hist[i], v);
  }
}

// 3. ------------------------------------------------------------------------------
__global__ void kmap_plan(const uint32_t* hist, int npass, int64_t N, KmapStatus* st) {
  __shared__ int constant_pass[kMaxPasses];
  if (threadIdx.x < kMaxPasses) constant_pass[threadIdx.x] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < npass * 256; i += blockDim.x)
    if (hist[i] == static_cast<uint64_t>(N)) constant_pass[i / 256] = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    int buf = 0;
    for (int p = 0; p < kMaxPasses; ++p) {
      const bool active = p < npass && !constant_pass[p];
      st->plan[p] = active ? (2 | buf) : 0;
      if (active) buf ^= 1;
    }
    st->plan[kMaxPasses] = buf;
  }
}

// 4a. per-block digit counts, digit-major: cnt[d * nblk + blk] -------------------------
__global__ void __launch_bounds__(kSortThreads) kmap_sort_count(
    const unsigned long long* __restrict__ mk0, const unsigned long long* __restrict__ mk1,
    int64_t N, int pass, int64_t nblk, uint32_t* __restrict__ cnt, const KmapStatus* st) {
  const int plan = st->plan[pass];
  if (!(plan & 2)) return;
  const unsigned long long* src = (plan & 1) ? mk1 : mk0;
  __shared__ uint32_t sh[256];
  sh[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = blockIdx.x * int64_t(kSortTile);
  for (int r = 0; r < kSortItems; ++r) {
    const int64_t e = base + r * kSortThreads + threadIdx.x;
    if (e < N) atomicAdd(&sh[(src[e] >> (8 * pass)) & 255u], 1u);
  }
  __syncthreads();
  cnt[threadIdx.x * nblk + blockIdx.x] = sh[threadIdx.x];
}

// 4b. one block per digit: exclusive scan over blocks plus the digit's base --------
__global__ void __launch_bounds__(256) kmap_sort_scan(const uint32_t* __restrict__ hist, int pass,
                                                      int64_t nblk, uint32_t* __restrict__ cnt,
                                                      const KmapStatus* st) {
  if (!(st->plan[pass] & 2)) return;
  const int d = blockIdx.x;
  __shared__ uint32_t warp_sums[8];
  __shared__ uint32_t carry;
  // base = sum of the histogram bins below d
  uint32_t v = threadIdx.x < static_cast<unsigned>(d) ? hist[pass * 256 + threadIdx.x] : 0u;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t s = 0;
    for (int w = 0; w < 8; ++w) s += warp_sums[w];
    carry = s;
  }
  __syncthreads();
  uint32_t* row = cnt + d * nblk;
  for (int64_t b0 = 0; b0 < nblk; b0 += 256) {
    const int64_t b = b0 + threadIdx.x;
    const uint32_t x = b < nblk ? row[b] : 0u;
    // block-wide inclusive scan of x
    uint32_t incl = x;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if ((threadIdx.x & 31) >= o) incl += y;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 31) warp_sums[threadIdx.x >> 5] = incl;
    __syncthreads();
    uint32_t wpre = 0;
    for (int w = 0; w < static_cast<int>(threadIdx.x >> 5); ++w) wpre += warp_sums[w];
    const uint32_t c0 = carry;
    if (b < nblk) row[b] = c0 + wpre + incl - x;
    __syncthreads();
    if (threadIdx.x == 255) carry = c0 + wpre + incl;
    __syncthreads();
  }
}

// 4c. stable scatter: rank inside the tile = earlier warps + earlier rounds + earlier lanes
__global__ void __launch_bounds__(kSortThreads) kmap_sort_scatter(
    unsigned long long* mk0, unsigned long long* mk1, int32_t* ix0, int32_t* ix1, int64_t N,
    int pass, int64_t nblk, const uint32_t* __restrict__ cnt, const KmapStatus* st) {
  const int plan = st->plan[pass];
  if (!(plan & 2)) return;
  const unsigned long long* src = (plan & 1) ? mk1 : mk0;
  unsigned long long* dst = (plan & 1) ? mk0 : mk1;
  const int32_t* isrc = (plan & 1) ? ix1 : ix0;
  int32_t* idst = (plan & 1) ? ix0 : ix1;
  constexpr int kWarps = kSortThreads / 32;
  constexpr int kPerWarp = kSortTile / kWarps;           // 512
  constexpr int kRounds = kPerWarp / 32;                 // 16
  __shared__ uint32_t wcnt[kWarps][257];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kWarps * 257; i += kSortThreads) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  const int64_t base = blockIdx.x * int64_t(kSortTile) + warp * kPerWarp;
  unsigned long long key[kRounds];
  int32_t row[kRounds];
  uint32_t rank[kRounds];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t e = base + r * 32 + lane;
    const bool valid = e < N;
    key[r] = valid ? src[e] : 0ull;
    row[r] = valid ? isrc[e] : 0;
    const uint32_t d = valid ? static_cast<uint32_t>((key[r] >> (8 * pass)) & 255u) : 256u;
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const uint32_t before = __popc(peers & lt_mask);
    const uint32_t prior = wcnt[warp][d];
    __syncwarp();
    if (before == 0) wcnt[warp][d] = prior + __popc(peers);
    __syncwarp();
    rank[r] = prior + before;
  }
  __syncthreads();
  {   // exclusive scan over warps, one thread per digit
    const int d = threadIdx.x;
    uint32_t run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t c = wcnt[w][d];
      wcnt[w][d] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t e = base + r * 32 + lane;
    if (e < N) {
      const uint32_t d = static_cast<uint32_t>((key[r] >> (8 * pass)) & 255u);
      const int64_t pos =
          int64_t(cnt[d * nblk + blockIdx.x]) + wcnt[warp][d] + rank[r];
      if (pos < N) {
        dst[pos] = key[r];
        idst[pos] = row[r];
      } else {
        atomicOr(const_cast<int*>(&st->flags), kFlagInternal);
      }
    }
  }
}

// 5. ------------------------------------------------------------------------------
__global__ void kmap_insert(const unsigned long long* __restrict__ keys,
                            const int32_t* __restrict__ ix0, const int32_t* __restrict__ ix1,
                            int64_t N, Slot* table, unsigned long long mask, int max_probe,
                            int32_t* __restrict__ order, KmapStatus* st) {
  const int32_t* sorted = (st->plan[kMaxPasses] & 1) ? ix1 : ix0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t s = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; s < N; s += stride) {
    const int32_t i = sorted[s];
    if (static_cast<uint64_t>(i) >= static_cast<uint64_t>(N)) {
      atomicOr(&st->flags, kFlagInternal);
      continue;
    }
    if (order) order[s] = i;
    const unsigned long long key = keys[i];
    unsigned long long h = home_slot(key, mask);
    int probe = 0;
    for (; probe < max_probe; ++probe) {
      const unsigned long long prev = atomicCAS(&table[h].key, kEmptyKey, key);
      if (prev == kEmptyKey) {
        table[h].row = i;
        break;
      }
      if (prev == key) {
        atomicOr(&st->flags, kFlagDup);
        atomicMin(&st->bad_row, static_cast<long long>(i));
        break;
      }
      h = (h + 1) & mask;
    }
    if (probe == max_probe) atomicOr(&st->flags, kFlagFull);
  }
}

// 6. ------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) kmap_probe(const int4* __restrict__ coords, int64_t N,
                                                  int res, const Slot* __restrict__ table,
                                                  unsigned long long mask, int max_probe,
                                                  int32_t* __restrict__ nbr, KmapStatus* st) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  bool full = false;
  for (int64_t v0 = warp_global * 32; v0 < N; v0 += nwarps * 32) {
    int4 mine = make_int4(0, 0, 0, 0);
    if (v0 + lane < N) mine = coords[v0 + lane];
    const int64_t nv = (N - v0) < 32 ? (N - v0) : 32;
#pragma unroll 1
    for (int t = 0; t < 27; ++t) {
      const int p = t * 32 + lane;          // flat (voxel, offset) index inside the warp's rows
      const int vv = p / 27;
      const int k = p - vv * 27;
      const int b = __shfl_sync(0xffffffffu, mine.x, vv);
      const int z = __shfl_sync(0xffffffffu, mine.y, vv) + (k / 9) - 1;
      const int y = __shfl_sync(0xffffffffu, mine.z, vv) + ((k / 3) % 3) - 1;
      const int x = __shfl_sync(0xffffffffu, mine.w, vv) + (k % 3) - 1;
      if (vv < nv) {
        int32_t found = -1;
        if (static_cast<unsigned>(z) < static_cast<unsigned>(res) &&
            static_cast<unsigned>(y) < static_cast<unsigned>(res) &&
            static_cast<unsigned>(x) < static_cast<unsigned>(res)) {
          const unsigned long long key = pack_key(b, z, y, x);
          unsigned long long h = home_slot(key, mask);
          int probe = 0;
          for (; probe < max_probe; ++probe) {
            const ulonglong2 s = __ldg(reinterpret_cast<const ulonglong2*>(table + h));
            if (s.x == key) {
              found = static_cast<int32_t>(s.y & 0xFFFFFFFFull);
              break;
            }
            if (s.x == kEmptyKey) break;
            h = (h + 1) & mask;
          }
          if (probe == max_probe) full = true;
        }
        nbr[v0 * 27 + p] = found;
      }
    }
  }
  if (full) atomicOr(&st->flags, kFlagFull);
}

int grid_for(int64_t work, int threads, int per_sm) {
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = int64_t(num_sms()) * per_sm;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
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

int kmap_build(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr, int32_t* order,
               int64_t hash_capacity, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (N < 0 || N > 0x7FFFFFFFll) {
    set_error("subm3d_build_kmap: N=%lld outside [0, 2^31)", (long long)N);
    return SUBM3D_ERR_ARG;
  }
  if (res < 1 || res > SUBM3D_MAX_RES) {
    set_error("subm3d_build_kmap: res=%d outside [1, %d]", res, SUBM3D_MAX_RES);
    return SUBM3D_ERR_ARG;
  }
  if (hash_capacity != 0 && (hash_capacity < 8 || (hash_capacity & (hash_capacity - 1)) ||
                             hash_capacity > (int64_t(1) << 40))) {
    set_error("subm3d_build_kmap: hash_capacity=%lld is not 0 or a power of two in [8, 2^40]",
              (long long)hash_capacity);
    return SUBM3D_ERR_ARG;
  }
  if (N == 0) return SUBM3D_OK;
  if (!coords || !nbr || !workspace) {
    set_error("subm3d_build_kmap: NULL pointer (coords=%p nbr=%p workspace=%p)", (const void*)coords,
              (void*)nbr, workspace);
    return SUBM3D_ERR_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(coords) & 15) || (reinterpret_cast<uintptr_t>(nbr) & 15) ||
      (order && (reinterpret_cast<uintptr_t>(order) & 15))) {
    set_error("subm3d_build_kmap: coords=%p nbr=%p order=%p must be 16-byte aligned",
              (const void*)coords, (void*)nbr, (void*)order);
    return SUBM3D_ERR_ARG;
  }
  const int64_t cap = hash_capacity > 0 ? hash_capacity : default_hash_capacity(N);
  const Layout L = make_layout(N, cap);
  if (reinterpret_cast<uintptr_t>(workspace) & 255) {
    set_error("subm3d_build_kmap: workspace=%p must be 256-byte aligned", workspace);
    return SUBM3D_ERR_WORKSPACE;
  }
  if (ws_bytes < L.total) {
    set_error("subm3d_build_kmap: workspace of %zu bytes, need %zu for N=%lld", ws_bytes, L.total,
              (long long)N);
    return SUBM3D_ERR_WORKSPACE;
  }
  char* ws = static_cast<char*>(workspace);
  KmapStatus* st = reinterpret_cast<KmapStatus*>(ws + L.status);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(ws + L.keys);
  unsigned long long* mk0 = reinterpret_cast<unsigned long long*>(ws + L.mk0);
  unsigned long long* mk1 = reinterpret_cast<unsigned long long*>(ws + L.mk1);
  int32_t* ix0 = reinterpret_cast<int32_t*>(ws + L.ix0);
  int32_t* ix1 = reinterpret_cast<int32_t*>(ws + L.ix1);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + L.cnt);
  Slot* table = reinterpret_cast<Slot*>(ws + L.table);

  int bits = 1;
  while ((1 << bits) < res) ++bits;
  const int npass = (3 * bits + 16 + 7) / 8;
  const unsigned long long mask = static_cast<unsigned long long>(cap - 1);
  const int max_probe = cap < kMaxProbe ? static_cast<int>(cap) : kMaxProbe;
  const int4* c4 = reinterpret_cast<const int4*>(coords);

  kmap_init<<<grid_for(cap, 256, 8), 256, 0, stream>>>(st, hist, table, cap);
  SUBM3D_LAUNCHED("kmap_init");
  kmap_pack<<<grid_for(N, 256, 4), 256, 0, stream>>>(c4, N, res, bits, npass, keys, mk0, ix0,
                                                     hist, st);
  SUBM3D_LAUNCHED("kmap_pack");
  kmap_plan<<<1, 256, 0, stream>>>(hist, npass, N, st);
  SUBM3D_LAUNCHED("kmap_plan");
  const int nblk = static_cast<int>(L.nblk);
  for (int p = 0; p < npass; ++p) {
    kmap_sort_count<<<nblk, kSortThreads, 0, stream>>>(mk0, mk1, N, p, L.nblk, cnt, st);
    SUBM3D_LAUNCHED("kmap_sort_count");
    kmap_sort_scan<<<256, 256, 0, stream>>>(hist, p, L.nblk, cnt, st);
    SUBM3D_LAUNCHED("kmap_sort_scan");
    kmap_sort_scatter<<<nblk, kSortThreads, 0, stream>>>(mk0, mk1, ix0, ix1, N, p, L.nblk, cnt, st);
    SUBM3D_LAUNCHED("kmap_sort_scatter");
  }
  kmap_insert<<<grid_for(N, 256, 8), 256, 0, stream>>>(keys, ix0, ix1, N, table, mask, max_probe,
                                                       order, st);
  SUBM3D_LAUNCHED("kmap_insert");
  kmap_probe<<<grid_for(N * 8, 256, 8), 256, 0, stream>>>(c4, N, res, table, mask, max_probe, nbr,
                                                          st);
  SUBM3D_LAUNCHED("kmap_probe");

  KmapStatus host;
  SUBM3D_CUDA_TRY(cudaMemcpyAsync(&host, st, sizeof(host), cudaMemcpyDeviceToHost, stream));
  SUBM3D_CUDA_TRY(cudaStreamSynchronize(stream));
  if (host.flags & kFlagInternal) {
    set_error("subm3d_build_kmap: internal error (sort produced an index outside [0, N))");
    return SUBM3D_ERR_DEVICE;
  }
  if (host.flags & kFlagCoord) {
    set_error("subm3d_build_kmap: coordinate row %lld outside 0<=b<=%d, 0<=z,y,x<%d",
              host.bad_row, SUBM3D_MAX_BATCH, res);
    return SUBM3D_ERR_COORD_RANGE;
  }
  if (host.flags & kFlagDup) {
    set_error("subm3d_build_kmap: duplicate coordinate (row %lld repeats an earlier key)",
              host.bad_row);
    return SUBM3D_ERR_DUPLICATE;
  }
  if (host.flags & kFlagFull) {
    set_error("subm3d_build_kmap: hash probe limit %d exceeded (capacity %lld, N=%lld)", max_probe,
              (long long)cap, (long long)N);
    return SUBM3D_ERR_HASH_FULL;
  }
  return SUBM3D_OK;
}

}  // namespace subm3d
