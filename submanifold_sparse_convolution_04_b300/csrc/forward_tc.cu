// Forward pass on the 5th-generation tensor cores (tcgen05): implicit gather-GEMM,
// output-stationary, bf16 in / fp32 accumulate in tensor memory.
//
// out[i, o] = bias[o] + sum_k sum_c W[o, kz, ky, kx, c] * feats[nbr[i, k], c]
// (submanifold convolution, kernel 3, stride 1, no padding, "pixal3d_mrp_mlx
// README" scope table; weight [O, kz, ky, kx, I], channels-last features, same
// README's commit header).
//
// One persistent CTA per SM loops over tiles of 128 output rows. For each tile the
// reduction runs over 27 offsets x ceil(I / 64) channel chunks; every (offset,
// chunk) step is one pipeline stage in shared memory:
//   A = the 128 gathered neighbour rows, 64 channels each (16 KB), in the
//       128-byte-swizzled K-major layout the tensor core reads, written either
//       - by tensor-copy gathers (cp.async.bulk.tensor tile::gather4: four rows of 64
//         channels per copy, half of an 8-row swizzle group; an absent neighbour is
//         the row coordinate -1, outside the feature tensor, which the copy fills
//         with zeros) when I is a multiple of 64: one producer warp per ring slot, a
//         lane per four rows, the stage's bytes counted on its barrier;
//       - or by 16-byte cp.async (an absent neighbour zero-fills and reads nothing),
//         groups of four producer warps (below);
//   B = W_k[:, chunk] = weight[:, kz, ky, kx, chunk], an [O x 64] K-major tile (I is
//       contiguous in the checkpoint layout, so no transpose), fetched by TMA with
//       the same 128-byte swizzle; out-of-range rows/columns are zero-filled. It sits
//       in the stage's own slot, fetched with the rows, except with TMA gathers and
//       O > 128, where the taps have a three-slot ring of their own (see Cfg).
// The row gathers are many small independent loads, and one warp can keep only a
// few kilobytes of cp.async in flight, so the gather rate grows with the number of
// warps issuing them, not with the depth of one warp's queue. The producers are
// therefore G groups of four warps (G = 6 for O <= 128): stage g belongs to group
// g mod G, and each group owns its own slots of the shared-memory ring, so G
// stages are gathered at once by 4G warps. Each producer thread fetches its eight
// nbr entries for its group's next stage while the current stage's copies are in
// flight (read-only loads, cached in L1), and the MMA thread asks L2 to prefetch
// the next tile's 13.8 KB nbr block when it starts a tile. A producer marks its
// stage full with cp.async.mbarrier.arrive.noinc (the slot counts as full the
// moment its rows land; no producer blocks on its own copies); the MMA thread
// orders those generic-proxy writes before its tensor-core reads with
// fence.proxy.async after the barrier wait.
// The MMA warp runs converged and one elected lane issues a stage's tcgen05.mma
// instructions (M = 128, N = round_up(O, 16), K = 16 each, up to four per stage) from a
// single asm block with a separate descriptor register per instruction: an MMA
// reads its register operands after issue, so reusing one register for the next
// instruction's descriptor serialises the MMAs (about 300 cycles each instead of
// 85 at N = 64 or 128 at N = 256). tcgen05.commit then frees the stage. Two
// accumulators (double-buffered tensor memory) let four epilogue warps drain tile t
// (tcgen05.ld, 8 columns at a time -> + bias [+ residual row, activation: the fused
// block epilogue] -> bf16 round-to-nearest-even -> one 16-byte store per 8 outputs)
// while the tensor core works on tile t + 1.
//
// Warp roles: warps 0 .. 4G-1 (cp.async) or 0 .. G-1 (TMA gathers) producers (the
// first thread of each group also issues its stages' weight TMA when the tap shares
// the stage's slot), then, with the taps' own ring, one loader warp, then the warp that
// allocates tensor memory and issues the MMAs (one lane), then four epilogue warps
// (warp w reads tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31).
// Every mbarrier wait is bounded (kWaitLimitNs); a wait that runs out sets the
// device error word, stops the CTA's pipeline, drains what is in flight and
// releases tensor memory before the CTA exits.
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace subm3d {

namespace {

constexpr int kBM = 128;          // output rows per tile (tensor-memory lanes)
constexpr int kKC = 64;           // channels per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxGroups = 6;     // producer groups of four warps
constexpr int kGroupThreads = 128;

// TG: the rows gathered by TMA (tile::gather4, four rows per copy, one producer warp per
// ring slot); otherwise by cp.async (groups of four producer warps). Each stage's weight
// tap goes into the stage's own B slot, fetched with its rows -- except for taps wider
// than 128 rows with TMA gathers (SPLIT): there a 32 KB tap per slot would leave room
// for only four slots, so the taps get a ring of three slots of their own, filled in
// stage order by a loader warp (a tap is needed only when its stage's MMAs issue, and
// at that width a stage's MMAs take long enough to cover the tap's fetch), and the rows
// get the rest of the shared memory (eight slots). At 128 rows and below the shorter
// stages need the taps further ahead, and the joint slots are faster.
template <int NMMA, bool TG>
struct Cfg {
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = NMMA * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kMisc = 1024 /*alignment slack*/ + 512 /*barriers*/ + 4 * 256 /*bias*/;
  static constexpr bool kSplit = TG && NMMA > 128;
  static constexpr int kSplitBSlots = 3;
  static constexpr int kFit = kSplit ? (kSmemLimit - kMisc - kSplitBSlots * kBBytes) / kABytes
                                     : (kSmemLimit - kMisc) / kStageBytes;
  static constexpr int kMaxG = TG ? 16 : kMaxGroups;
  static constexpr int kGroups = kFit < kMaxG ? kFit : kMaxG;
  static constexpr int kSlots = kFit / kGroups;            // ring slots per group
  static constexpr int kStages = kGroups * kSlots;          // A slots
  static constexpr int kBSlots = kSplit ? kSplitBSlots : kStages;   // B slots
  static constexpr int kNB = kSplit ? kBSlots : 0;          // barriers of the weight ring
  static constexpr int kGroupWarps = TG ? 1 : 4;
  static constexpr int kLoadWarp = kGroupWarps * kGroups;   // SPLIT: the weight loader
  static constexpr int kMmaWarp = kLoadWarp + (kSplit ? 1 : 0);
  static constexpr int kEpiWarp0 = kMmaWarp + 1;
  static constexpr int kThreads = 32 * (kEpiWarp0 + 4);
  // one tile's accumulator: NMMA columns, placed at a power-of-two column stride
  static constexpr int kBufCols = NMMA <= 16 ? 16 : NMMA <= 32 ? 32 : NMMA <= 64 ? 64
                                : NMMA <= 128 ? 128 : 256;
  static constexpr int kTmemCols = 2 * kBufCols < 32 ? 32 : 2 * kBufCols;
  static constexpr int kSmemBytes = kMisc + kStages * kABytes + kBSlots * kBBytes;
  static_assert(kGroups >= 3, "too few producer groups");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory");
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "tensor memory");
  static_assert(kThreads <= 1024, "block too large");
  static_assert(8 * (2 * kStages + 2 * kNB + 5) + 8 <= 512, "barrier area too small");
};

struct Params {
  const __nv_bfloat16* feats;
  const int32_t* nbr;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  const __nv_bfloat16* residual;   // [N, O] or NULL (may equal out)
  int act;                         // subm3d_act
  int64_t N;
  int I, O;
  int nchunks;
  int ntiles;
  int* err;
  const int32_t* perm;             // tile plan: plan row -> output row, or NULL (identity)
  const uint32_t* tmask;           // tile plan: offsets present per tile, or NULL (all 27)
};

// Offsets a tile runs: its plan mask (the centre always included), or all 27.
__device__ __forceinline__ uint32_t tile_mask(const Params& p, int tile) {
  return p.tmask ? ((__ldg(p.tmask + tile) & 0x7FFFFFFu) | (1u << 13)) : 0x7FFFFFFu;
}
// The i-th (from 0) set bit of m: a binary search over popcounts of halves, without a
// loop over the bits below it.
__device__ __forceinline__ int nth_offset(uint32_t m, int i) {
  int pos = 0;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const int c = __popc((m >> pos) & ((1u << w) - 1u));
    if (i >= c) {
      i -= c;
      pos += w;
    }
  }
  return pos;
}

// Walks a CTA's stages in order: stage g is step g - g0 of local tile lt, a step being
// one (offset, channel chunk); a tile has popcount(mask) x nchunks steps.
struct StageCursor {
  int lt = 0;
  uint32_t g0 = 0, steps = 0, mask = 0;
  __device__ __forceinline__ void start(const Params& p, int ntl) {
    lt = 0;
    g0 = 0;
    if (ntl > 0) {
      mask = tile_mask(p, blockIdx.x);
      steps = __popc(mask) * static_cast<uint32_t>(p.nchunks);
    }
  }
  // Moves to stage g (never backwards); false past the CTA's last stage.
  __device__ __forceinline__ bool seek(const Params& p, int ntl, uint32_t g) {
    while (lt < ntl && g >= g0 + steps) {
      g0 += steps;
      ++lt;
      if (lt < ntl) {
        mask = tile_mask(p, blockIdx.x + lt * gridDim.x);
        steps = __popc(mask) * static_cast<uint32_t>(p.nchunks);
      }
    }
    return lt < ntl;
  }
};

// Stage g of a cursor as (offset index in its tile, channel chunk). A group's stages
// advance by G at a time: inside one tile that is a fixed step (dq offsets, dr chunks,
// with carry), so only the first stage of a tile divides.
struct StagePos {
  int lt = -1, oi = 0, c = 0;
  uint32_t g = 0;
  __device__ __forceinline__ void locate(const StageCursor& cur, uint32_t gg, uint32_t G,
                                         int nchunks, int dq, int dr) {
    if (cur.lt == lt && gg == g + G) {
      c += dr;
      oi += dq;
      if (c >= nchunks) {
        c -= nchunks;
        ++oi;
      }
    } else {
      const uint32_t kc = gg - cur.g0;
      oi = static_cast<int>(kc / static_cast<uint32_t>(nchunks));
      c = static_cast<int>(kc - static_cast<uint32_t>(oi) * static_cast<uint32_t>(nchunks));
    }
    lt = cur.lt;
    g = gg;
  }
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);          // start address
  d |= static_cast<uint64_t>(1) << 16;                            // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                    // stride offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                            // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                            // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both K-major.
template <int NMMA>
__device__ __forceinline__ uint32_t make_idesc() {
  return (1u << 4)                                  // D format fp32
         | (1u << 7)                                // A format bf16
         | (1u << 10)                               // B format bf16
         | (static_cast<uint32_t>(NMMA >> 3) << 17)  // N / 8
         | (static_cast<uint32_t>(kBM >> 4) << 24);  // M / 16
}

// Bounded wait used only while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Warp-uniform bounded wait: every lane polls the barrier; the warp proceeds only if
// all lanes saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// One stage's MMAs, K = 16 each (ksteps of them, 1..4), issued by one elected lane of a
// converged warp. K step kk starts 32 bytes further into both 128-byte-swizzled
// tiles, i.e. +2 in the descriptors' address field. The first MMA accumulates only if
// `acc` is set; the later ones always do. Every MMA gets its own descriptor
// registers (see the file comment).
__device__ __forceinline__ void mma_stage(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          int ksteps, uint32_t acc) {
  const uint64_t a1 = a + 2, a2 = a + 4, a3 = a + 6;
  const uint64_t b1 = b + 2, b2 = b + 4, b3 = b + 6;
#define SUBM3D_MMA_HEAD                                                   \
  "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %9, 0;\n\t"                    \
  "elect.sync _|e, 0xffffffff;\n\t"                                       \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %10, p;\n\t"
#define SUBM3D_MMA(A, B) "@e tcgen05.mma.cta_group::1.kind::f16 [%0], " A ", " B ", %10, 1;\n\t"
#define SUBM3D_MMA_ARGS                                                                  \
  "r"(d), "l"(a), "l"(a1), "l"(a2), "l"(a3), "l"(b), "l"(b1), "l"(b2), "l"(b3), "r"(acc), \
      "r"(idesc)
  switch (ksteps) {
    case 4:
      asm volatile(SUBM3D_MMA_HEAD SUBM3D_MMA("%2", "%6") SUBM3D_MMA("%3", "%7")
                       SUBM3D_MMA("%4", "%8") "}" ::SUBM3D_MMA_ARGS
                   : "memory");
      break;
    case 3:
      asm volatile(SUBM3D_MMA_HEAD SUBM3D_MMA("%2", "%6") SUBM3D_MMA("%3", "%7") "}" ::SUBM3D_MMA_ARGS
                   : "memory");
      break;
    case 2:
      asm volatile(SUBM3D_MMA_HEAD SUBM3D_MMA("%2", "%6") "}" ::SUBM3D_MMA_ARGS : "memory");
      break;
    default:
      asm volatile(SUBM3D_MMA_HEAD "}" ::SUBM3D_MMA_ARGS : "memory");
      break;
  }
#undef SUBM3D_MMA_HEAD
#undef SUBM3D_MMA
#undef SUBM3D_MMA_ARGS
}

// tcgen05.commit from one elected lane of a converged warp.
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// The eight nbr entries producer thread (rsub, q) needs for a stage of tile-row
// block row0 at offset k: rows rsub + 16 m, m = 0..7 (-1 past N). An entry outside
// [-1, N) is reported through `bad` and treated as absent.
__device__ __forceinline__ void load_rows(const Params& p, int64_t row0, int k, int rsub,
                                          int32_t (&j)[8], bool& bad) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int64_t row = row0 + rsub + 16 * m;
    int32_t v = -1;
    if (row < p.N) {
      v = __ldg(p.nbr + row * 27 + k);
      if (v < -1 || v >= p.N) {
        bad = true;
        v = -1;
      }
    }
    j[m] = v;
  }
}

// Rows 4 lane + m (m = 0..3) of a TMA-gathered stage of tile-row block row0 at offset k:
// their input rows, -1 (a coordinate outside the feature tensor: the copy fills zeros)
// for an absent neighbour or a row past N. An entry outside [-1, N) is reported through
// `bad` and treated as absent.
__device__ __forceinline__ void load_rows4(const Params& p, int64_t row0, int k, int lane,
                                           int32_t (&j)[4], bool& bad) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int64_t row = row0 + 4 * lane + m;
    int32_t v = -1;
    if (row < p.N) {
      v = __ldg(p.nbr + row * 27 + k);
      if (v < -1 || v >= p.N) {
        bad = true;
        v = -1;
      }
    }
    j[m] = v;
  }
}

// Four rows (y0..y3) of 64 channels from column x of a 2D tensor map into shared memory
// at dst (128-byte swizzle, rows 128 bytes apart), completing on `bar` by bytes.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, const int32_t (&y)[4]) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y[0]), "r"(y[1]), "r"(y[2]), "r"(y[3]),
      "r"(bar)
      : "memory");
}

template <int NMMA, bool TG>
__global__ void __launch_bounds__(Cfg<NMMA, TG>::kThreads, 1)
    fwd_tc(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap fmap,
           const Params p) {
  using C = Cfg<NMMA, TG>;
  constexpr int S = C::kStages;
  constexpr int G = C::kGroups;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  constexpr int SB = C::kBSlots;
  const uint32_t sA = base;                              // S x 16 KB
  const uint32_t sB = base + S * C::kABytes;             // SB x NMMA*128 B
  uint8_t* misc = base_ptr + S * C::kABytes + SB * C::kBBytes;
  // barriers: full[S], empty[S], (SPLIT) bfull[SB], bempty[SB], accf[2], acce[2], drain
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t bfull0 = empty0 + 8 * S;
  const uint32_t bempty0 = bfull0 + 8 * C::kNB;
  const uint32_t accf0 = bempty0 + 8 * C::kNB;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (2 * S + 2 * C::kNB + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* bias_sm = reinterpret_cast<float*>(misc + 512);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // tiles of this CTA: blockIdx.x + t * gridDim.x, t < ntl; stages per tile: spt
  const int ntl = (p.ntiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                  static_cast<int>(gridDim.x);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      // cp.async: a group's noinc arrivals + the weight TMA's; TMA gathers: one arrival
      // with the stage's row bytes
      mbar_init(full0 + 8 * s, TG ? 1 : kGroupThreads + 1);
      mbar_init(empty0 + 8 * s, 1);                  // one tcgen05.commit
    }
    for (int b = 0; b < C::kNB; ++b) {
      mbar_init(bfull0 + 8 * b, 1);                  // the loader's arrival with the tap's bytes
      mbar_init(bempty0 + 8 * b, 1);                 // one tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&wmap);
    if (TG) tma_prefetch_desc(&fmap);
  }
  if (warp >= C::kEpiWarp0) {
    for (int o = tid - C::kEpiWarp0 * 32; o < NMMA; o += 128)
      bias_sm[o] = (p.bias && o < p.O) ? __bfloat162float(p.bias[o]) : 0.f;
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (TG && warp < C::kLoadWarp) {
    // ----------------------------------------------- producers, rows gathered by TMA
    // warp grp owns the stages g = grp (mod G); lane l copies rows 4 l .. 4 l + 3 of a
    // stage with one gather4 into their 128-byte-swizzled places (rows 4 l .. 4 l + 3 of
    // the K-major A tile: half of an 8-row swizzle group, 512 bytes), lane 0 first
    // announcing the stage's bytes (and, with joint slots, fetching its weight tap)
    const int grp = warp;
    bool bad = false, aborted = false;
    uint32_t last = 0;
    int32_t jn[4];
    StageCursor cur, nxt;
    StagePos pc, pn;
    const int dq = G / p.nchunks, dr = G % p.nchunks;
    cur.start(p, ntl);
    nxt.start(p, ntl);
    if (nxt.seek(p, ntl, grp)) {
      pn.locate(nxt, grp, G, p.nchunks, dq, dr);
      load_rows4(p, int64_t(blockIdx.x + nxt.lt * gridDim.x) * kBM, nth_offset(nxt.mask, pn.oi),
                 lane, jn, bad);
    }
    for (uint32_t g = grp; cur.seek(p, ntl, g); g += G) {
      pc.locate(cur, g, G, p.nchunks, dq, dr);
      const int c = pc.c;
      const int k = nth_offset(cur.mask, pc.oi);
      int32_t j[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) j[m] = jn[m];
      if (nxt.seek(p, ntl, g + G)) {
        pn.locate(nxt, g + G, G, p.nchunks, dq, dr);
        load_rows4(p, int64_t(blockIdx.x + nxt.lt * gridDim.x) * kBM, nth_offset(nxt.mask, pn.oi),
                   lane, jn, bad);
      }
      const uint32_t s = g % S;
      const uint32_t ph = (g / S) & 1u;
      if (!warp_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) {
        aborted = true;
        break;
      }
      if (lane == 0) {
        if (C::kSplit) {
          mbar_arrive_expect_tx(full0 + 8 * s, C::kABytes);
        } else {
          mbar_arrive_expect_tx(full0 + 8 * s, C::kABytes + C::kBBytes);
          tma_load_3d(sB + s * C::kBBytes, &wmap, full0 + 8 * s, c * kKC, k, 0);
        }
      }
      __syncwarp();
      tma_gather4(sA + s * C::kABytes + lane * 512, &fmap, full0 + 8 * s, c * kKC, j);
      last = g + G;
    }
    if (bad) atomicOr(p.err, kDevErrBadNbr);
    if (aborted && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, kDevErrTimeout);
      // no copy of this warp may still be landing in shared memory when the CTA exits
      // (without an abort the MMA warp has waited for every stage)
      for (uint32_t x = last >= static_cast<uint32_t>(S) ? last - S : 0u; x < last; ++x)
        if (x % G == static_cast<uint32_t>(grp)) drain_wait(full0 + 8 * (x % S), (x / S) & 1u);
    }
    __syncwarp();
  } else if (C::kSplit && warp == C::kLoadWarp) {
    // ----------------------------------------------- weight taps, in stage order (SPLIT)
    bool aborted = false;
    uint32_t last = 0;
    StageCursor cur;
    StagePos pc;
    const int dq = 1 / p.nchunks, dr = 1 % p.nchunks;
    cur.start(p, ntl);
    for (uint32_t g = 0; cur.seek(p, ntl, g); ++g) {
      pc.locate(cur, g, 1u, p.nchunks, dq, dr);
      const uint32_t b = g % SB;
      if (!warp_wait(bempty0 + 8 * b, ((g / SB) & 1u) ^ 1u, abort_flag)) {
        aborted = true;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bfull0 + 8 * b, C::kBBytes);
        tma_load_3d(sB + b * C::kBBytes, &wmap, bfull0 + 8 * b, pc.c * kKC,
                    nth_offset(cur.mask, pc.oi), 0);
      }
      __syncwarp();
      last = g + 1;
    }
    if (aborted && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, kDevErrTimeout);
      // no tap may still be landing in shared memory when the CTA exits
      for (uint32_t x = last >= static_cast<uint32_t>(SB) ? last - SB : 0u; x < last; ++x)
        drain_wait(bfull0 + 8 * (x % SB), (x / SB) & 1u);
    }
    __syncwarp();
  } else if (warp < C::kMmaWarp) {
    // ------------------------------------------------------------------ producers
    const int grp = warp >> 2;
    const int gt = tid & (kGroupThreads - 1);
    const int q = gt & 7;           // 16-byte column chunk inside the 128-byte row
    const int rsub = gt >> 3;       // rows rsub + 16 m, m = 0..7
    bool bad = false, aborted = false;
    uint32_t last = 0;              // one past the last stage this group issued
    int32_t jn[8];
    // cur: this group's stage; nxt: the one after it (its rows load a stage ahead)
    StageCursor cur, nxt;
    StagePos pc, pn;
    const int dq = G / p.nchunks, dr = G % p.nchunks;
    cur.start(p, ntl);
    nxt.start(p, ntl);
    if (nxt.seek(p, ntl, grp)) {
      pn.locate(nxt, grp, G, p.nchunks, dq, dr);
      load_rows(p, int64_t(blockIdx.x + nxt.lt * gridDim.x) * kBM, nth_offset(nxt.mask, pn.oi),
                rsub, jn, bad);
    }
    for (uint32_t g = grp; cur.seek(p, ntl, g); g += G) {
      pc.locate(cur, g, G, p.nchunks, dq, dr);
      const int c = pc.c;
      const int k = nth_offset(cur.mask, pc.oi);
      int32_t j[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) j[m] = jn[m];
      if (nxt.seek(p, ntl, g + G)) {   // next stage's rows: in flight while this stage is issued
        pn.locate(nxt, g + G, G, p.nchunks, dq, dr);
        load_rows(p, int64_t(blockIdx.x + nxt.lt * gridDim.x) * kBM, nth_offset(nxt.mask, pn.oi),
                  rsub, jn, bad);
      }
      const uint32_t s = g % S;
      const uint32_t ph = (g / S) & 1u;
      if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) {
        aborted = true;
        break;
      }
      if (gt == 0) {
        mbar_arrive_expect_tx(full0 + 8 * s, C::kBBytes);
        tma_load_3d(sB + s * C::kBBytes, &wmap, full0 + 8 * s, c * kKC, k, 0);
      }
      const int col = c * kKC + q * 8;
      const bool col_ok = col < p.I;
      const uint32_t a_stage = sA + s * C::kABytes;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int r = rsub + 16 * m;
        const uint32_t dst = a_stage + r * 128 + ((q ^ (r & 7)) << 4);
        const bool ok = col_ok && j[m] >= 0;
        const __nv_bfloat16* src = ok ? p.feats + int64_t(j[m]) * p.I + col : p.feats;
        cp_async_16(dst, src, ok ? 16u : 0u);
      }
      cp_async_arrive_noinc(full0 + 8 * s);   // stage s is full once these land
      last = g + G;
    }
    cp_async_wait_all();   // no gather of this thread is still landing when the CTA exits
    if (bad) atomicOr(p.err, kDevErrBadNbr);
    if (aborted) {
      *abort_flag = 1;
      atomicOr(p.err, kDevErrTimeout);
      if (gt == 0) {   // no weight TMA of this group may still be landing in shared memory
        for (uint32_t x = last >= static_cast<uint32_t>(S) ? last - S : 0u; x < last; ++x)
          if (x % G == static_cast<uint32_t>(grp)) drain_wait(full0 + 8 * (x % S), (x / S) & 1u);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------------ MMA issue
    const uint32_t idesc = make_idesc<NMMA>();
    uint32_t g = 0;
    bool aborted = false;
    for (int t = 0; t < ntl && !aborted; ++t) {
      if (t + 1 < ntl && lane == 0) {   // the next tile's nbr block into L2 while this tile runs
        const int64_t row1 = int64_t(blockIdx.x + (t + 1) * gridDim.x) * kBM;
        const int64_t rows = (p.N - row1) < kBM ? (p.N - row1) : kBM;
        const uint32_t bytes = static_cast<uint32_t>(rows * 108) & ~15u;
        if (bytes) bulk_prefetch_l2(p.nbr + row1 * 27, bytes);
      }
      const uint32_t buf = t & 1u;
      const uint32_t use = t >> 1;
      if (!warp_wait(acce0 + 8 * buf, (use & 1u) ^ 1u, abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * C::kBufCols;
      const uint32_t spt = __popc(tile_mask(p, blockIdx.x + t * gridDim.x)) *
                           static_cast<uint32_t>(p.nchunks);
      int c = 0;   // the stage's channel chunk, counted along (no division per stage)
      for (uint32_t kc = 0; kc < spt; ++kc, c = (c + 1 == p.nchunks) ? 0 : c + 1) {
        const uint32_t s = g % S;
        const uint32_t ph = (g / S) & 1u;
        const uint32_t b = C::kSplit ? g % SB : s;   // the stage's weight slot
        if (!warp_wait(full0 + 8 * s, ph, abort_flag) ||
            (C::kSplit && !warp_wait(bfull0 + 8 * b, (g / SB) & 1u, abort_flag))) {
          aborted = true;
          break;
        }
        fence_proxy_async_smem();
        tc_fence_after();
        const int rem = p.I - c * kKC;
        const int ksteps = rem >= kKC ? 4 : (rem + 15) / 16;
        mma_stage(d_tmem, sw128_desc(sA + s * C::kABytes), sw128_desc(sB + b * C::kBBytes), idesc,
                  ksteps, kc == 0 ? 0u : 1u);
        tc_commit_elect(empty0 + 8 * s);
        if (C::kSplit) tc_commit_elect(bempty0 + 8 * b);
        ++g;
      }
      if (!aborted) tc_commit_elect(accf0 + 8 * buf);
    }
    if (aborted) {
      if (lane == 0) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
      tc_commit_elect(drain);   // wait for every MMA already issued
      if (lane == 0) drain_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int lg = warp & 3;                  // tensor-memory lane group of this warp
    for (int t = 0; t < ntl; ++t) {
      const int tile = blockIdx.x + t * gridDim.x;
      const uint32_t buf = t & 1u;
      const uint32_t use = t >> 1;
      const int64_t prow = int64_t(tile) * kBM + lg * 32 + lane;   // row of the tile order
      int64_t row = prow;                                          // output row
      if (p.perm && prow < p.N) {
        row = __ldg(p.perm + prow);
        if (row < 0 || row >= p.N) {   // a plan row that names no input row: skipped
          atomicOr(p.err, kDevErrBadPlan);
          row = p.N;
        }
      }
      // the residual row travels to L2, and its first 16 bytes to registers, while this
      // warp waits for the accumulator
      const __nv_bfloat16* rrow = (p.residual && row < p.N) ? p.residual + row * p.O : nullptr;
      uint4 rnext = make_uint4(0, 0, 0, 0);
      if (rrow) {
        prefetch_row_l2(rrow, p.O * 2);
        rnext = ld_row16(rrow);
      }
      if (!mbar_wait(accf0 + 8 * buf, use & 1u, abort_flag)) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + buf * C::kBufCols;
      __nv_bfloat16* orow = p.out + row * p.O;
#pragma unroll 1
      for (int cc = 0; cc < NMMA / 8; ++cc) {   // 8 columns at a time
        uint32_t v[8];
        tmem_ld8(taddr + cc * 8, v);
        const uint4 rcur = rnext;   // the next group's residual loads during this one
        if (rrow && cc * 8 + 8 < p.O) rnext = ld_row16(rrow + cc * 8 + 8);
        tmem_ld_wait();
        if (cc == NMMA / 8 - 1) {
          tc_fence_before();
          mbar_arrive(acce0 + 8 * buf);
        }
        const int col0 = cc * 8;
        if (row < p.N && col0 < p.O) {
          // streaming store: the output is not read again here, the gathered rows are
          __stcs(reinterpret_cast<uint4*>(orow + col0),
                 epilogue8_bf16(v, bias_sm + col0, rrow != nullptr, rcur, p.act));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

template <int NMMA, bool TG>
int launch(const Params& prm, const __nv_bfloat16* weight, cudaStream_t stream) {
  using C = Cfg<NMMA, TG>;
  static PerDevice<bool> attr_set;
  const int arc = set_smem_limit_once(attr_set, reinterpret_cast<const void*>(fwd_tc<NMMA, TG>),
                                      C::kSmemBytes, "fwd_tc");
  if (arc != SUBM3D_OK) return arc;
  EncodeTiledFn encode = get_encode();
  if (!encode) {
    set_error("subm3d_forward: cuTensorMapEncodeTiled is not available from the driver");
    return SUBM3D_ERR_CUDA;
  }
  CUtensorMap map;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(prm.I), 27, static_cast<cuuint64_t>(prm.O)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(prm.I) * 2,
                                 static_cast<cuuint64_t>(prm.I) * 27 * 2};
  const cuuint32_t box[3] = {kKC, 1, NMMA};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(weight),
                            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("subm3d_forward: cuTensorMapEncodeTiled failed (%d) for weight=%p I=%d O=%d",
              static_cast<int>(r), (const void*)weight, prm.I, prm.O);
    return SUBM3D_ERR_CUDA;
  }
  // the feature rows for the TMA gathers: [N rows x I channels], boxes of one row of 64
  // channels, the same 128-byte swizzle as the A tile; a row coordinate outside [0, N)
  // reads zeros
  CUtensorMap fmap;
  std::memset(&fmap, 0, sizeof(fmap));
  if (TG) {
    const cuuint64_t fdims[2] = {static_cast<cuuint64_t>(prm.I), static_cast<cuuint64_t>(prm.N)};
    const cuuint64_t fstrides[1] = {static_cast<cuuint64_t>(prm.I) * 2};
    const cuuint32_t fbox[2] = {kKC, 1};
    const cuuint32_t festr[2] = {1, 1};
    const CUresult fr = encode(&fmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                               const_cast<__nv_bfloat16*>(prm.feats), fdims, fstrides, fbox, festr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (fr != CUDA_SUCCESS) {
      set_error("subm3d_forward: cuTensorMapEncodeTiled failed (%d) for feats=%p N=%lld I=%d",
                static_cast<int>(fr), (const void*)prm.feats, (long long)prm.N, prm.I);
      return SUBM3D_ERR_CUDA;
    }
  }
  const int grid = prm.ntiles < num_sms() ? prm.ntiles : num_sms();
  fwd_tc<NMMA, TG><<<grid, C::kThreads, C::kSmemBytes, stream>>>(map, fmap, prm);
  SUBM3D_LAUNCHED(TG ? "fwd_tc_tg" : "fwd_tc");
  return SUBM3D_OK;
}

}  // namespace

int forward_launch_tc(const __nv_bfloat16* feats, const int32_t* nbr, const __nv_bfloat16* weight,
                      const __nv_bfloat16* bias, __nv_bfloat16* out, int64_t N, int I, int O,
                      Epilogue epi, TilePlan plan, cudaStream_t stream) {
  const int64_t ntiles = (N + kBM - 1) / kBM;
  if (ntiles > 0x7FFFFFFFll) {
    set_error("subm3d_forward: N=%lld too large", (long long)N);
    return SUBM3D_ERR_UNSUPPORTED;
  }
  int* err = forward_error_word();
  if (!err) return SUBM3D_ERR_CUDA;
  Params prm{feats, nbr, bias, out, static_cast<const __nv_bfloat16*>(epi.residual), epi.act,
             N, I, O, (I + kKC - 1) / kKC, static_cast<int>(ntiles), err, plan.perm, plan.tmask};
  const int nmma = (O + 15) / 16 * 16;
  // The rows by TMA gathers when every channel chunk is whole (the copies' column start a
  // multiple of 64 channels, 128 bytes): on a B300, 433 us against 564 us with cp.async
  // at I = O = 128 (753 k voxels), and with the taps in a ring of their own 462 us
  // against 512 us at I = O = 256 (278 k voxels).
  const bool tg = I % kKC == 0 && N <= 0x7FFFFFFFll;
  switch (nmma) {
#define SUBM3D_CASE(n)                                                          \
  case n:                                                                       \
    return tg ? launch<n, true>(prm, weight, stream) : launch<n, false>(prm, weight, stream);
    SUBM3D_CASE(16) SUBM3D_CASE(32) SUBM3D_CASE(48) SUBM3D_CASE(64)
    SUBM3D_CASE(80) SUBM3D_CASE(96) SUBM3D_CASE(112) SUBM3D_CASE(128)
    SUBM3D_CASE(144) SUBM3D_CASE(160) SUBM3D_CASE(176) SUBM3D_CASE(192)
    SUBM3D_CASE(208) SUBM3D_CASE(224) SUBM3D_CASE(240) SUBM3D_CASE(256)
#undef SUBM3D_CASE
    default:
      set_error("subm3d_forward: O=%d outside the tensor-core kernel's range", O);
      return SUBM3D_ERR_UNSUPPORTED;
  }
}

}  // namespace subm3d
