// Forward pass for narrow layers (I <= 64, O <= 64, both multiples of 16): implicit
// gather-GEMM on the 5th-generation tensor cores with the gathered operand in
// tensor memory.
//
// out[i, o] = bias[o] + sum_k sum_c W[o, kz, ky, kx, c] * feats[nbr[i, k], c]
// (submanifold convolution, kernel 3, stride 1, no padding, "pixal3d_mrp_mlx
// README" scope table; weight [O, kz, ky, kx, I], channels-last features, same
// README's commit header).
//
// Why a second kernel: with the gathered rows staged in shared memory, every 128-row
// stage costs 48 KB of shared-memory traffic at O = 64 (16 KB of cp.async writes,
// most of them zero-fill, the MMA re-reading them, and the weight tile written and
// read), and the shared-memory port, not HBM, sets the pace. Here:
//   * the gathered rows reach a tensor-memory stage through registers, the row in the
//     lane of its output row, channels 2c and 2c+1 in column c, written by tcgen05.st;
//     an absent neighbour costs no load at all (zeros). Two forms of the gather:
//     - each lane loads its own row with four 32-byte read-only loads (six producer
//       groups): few instructions per row, but the L1 data pipe takes about eight passes
//       per row; the faster form for input-order tiles, which run all 27 offsets;
//     - a producer warp copies its 32 rows of an offset with coalesced 16-byte cp.async
//       copies (eight lanes per 128-byte row) into its own shared-memory staging area,
//       and each lane reads its own row back (four producer groups, a staging buffer
//       per offset of a stage): one L1 pass per row, more instructions per offset; the
//       faster form for the tiles of a plan, which run about half the offsets;
//   * tcgen05.mma reads A from tensor memory and only B, the stage's weight tap
//     W_k = weight[:, kz, ky, kx, :] ([O x 64] K-major, 128-byte swizzle, fetched by
//     TMA into the stage's weight slot), from shared memory;
//   * a loader warp copies each tile's 128 x 27 block of nbr (13.8 KB, contiguous)
//     into a double-buffered shared-memory ring with one bulk copy, a tile ahead, so
//     a producer reads its row's index with one conflict-free shared load (27 is
//     odd) instead of one 32-byte global sector per 4-byte index.
// Tensor memory (512 columns allocated): two accumulators of 64 columns (double buffer)
// and one A stage of 64 columns per producer group (six or four). A stage carries two
// offsets of the tile (consecutive offsets of its mask; the last may have one), because
// every stage costs the single MMA-issuing warp a barrier wait and a commit. Stage g of
// the CTA is filled by producer group g mod G (four warps, warp w writing lanes
// 32 (w % 4) .. + 31) into slot g mod G: each warp starts its rows of the stage's first
// offset (with staging, of both offsets) while the slot frees, stores the first and then
// the second; the group leader fetches both weight taps into the stage's weight slot by
// TMA. The stage is full when its four warps have arrived (after tcgen05.wait::st) and
// its weight bytes have landed.
// One elected lane of the MMA warp issues the stage's MMAs (M = 128, N = O, K = 16,
// up to four per offset) and frees the slot with tcgen05.commit. Four epilogue warps drain tile
// t (tcgen05.ld -> + bias [+ residual row, activation: the fused block epilogue] ->
// bf16 round-to-nearest-even -> 16-byte stores) while the tensor core works on tile t + 1.
//
// Every mbarrier wait is bounded (kWaitLimitNs); a wait that runs out sets the device
// error word, stops the CTA's pipeline, drains what is in flight and releases tensor
// memory before the CTA exits.
#include <mutex>

#include "common.cuh"

namespace subm3d {
namespace {

constexpr int kBM = 128;              // output rows per tile = tensor-memory lanes
constexpr int kOffCols = 32;          // one offset's row: 64 bf16 = 32 columns of 32 bits
constexpr int kStageCols = 2 * kOffCols;   // a stage holds two offsets (2p, 2p + 1)
constexpr int kAccCols = 64;          // one accumulator (N <= 64)
constexpr int kAColBase = 2 * kAccCols;
constexpr int kNbrTileBytes = kBM * 27 * 4;      // one tile's rows of nbr
constexpr int kRowsStaging = 32 * 128;           // a producer warp's 32 gathered rows
constexpr int kSmemLimit = 227 * 1024;

// Warp roles and pipeline depth of the two gather forms (see the file comment):
// STAGED, whole rows copied through a per-warp shared-memory staging area, four producer
// groups with two buffers per warp; otherwise each lane loads its own row into
// registers, six producer groups (more warps keep more loads in flight).
template <bool STAGED>
struct TmRoles {
  static constexpr int kGroups = STAGED ? 4 : 6;        // producer groups of four warps
  static constexpr int kStages = kGroups;               // A stages in tensor memory
  static constexpr int kProducerWarps = 4 * kGroups;
  static constexpr int kMmaWarp = kProducerWarps;
  static constexpr int kEpiWarp0 = kMmaWarp + 1;        // four warps: lane groups w % 4
  static constexpr int kNbrWarp = kEpiWarp0 + 4;
  static constexpr int kThreads = 32 * (kNbrWarp + 1);  // 704 staged, 960 otherwise
  static constexpr int kWarpStaging = STAGED ? 2 * kRowsStaging : 0;   // a buffer per offset
  static constexpr int kStagingBytes = kProducerWarps * kWarpStaging;
  // per-thread form: the epilogue warps' output rows pass through shared memory (32 rows
  // of up to 128 bytes per warp, a 16-byte pad per row) so that whole rows leave with
  // coalesced stores; the staged form has no room left for it
  static constexpr int kEpiPitch = 128 + 16;
  static constexpr int kEpiStagingBytes = STAGED ? 0 : 4 * 32 * kEpiPitch;
  static_assert(kAColBase + kStages * kStageCols <= 512, "tensor memory layout");
  static_assert(kStages % kGroups == 0, "slots per group");
  static_assert(((kEpiWarp0 & 3) + 0) >= 0, "epilogue warps cover the four lane groups");
};

template <int NMMA, bool STAGED>
struct TmCfg {
  using R = TmRoles<STAGED>;
  static constexpr int kTapBytes = NMMA * 128;               // one [NMMA x 64] weight tile
  static constexpr int kWBytes = R::kStages * 2 * kTapBytes;  // two taps per stage
  static constexpr int kUsed = 1024 /*alignment*/ + kWBytes + 2 * kNbrTileBytes +
                               512 /*barriers*/ + 256 * 4 /*bias*/ + R::kStagingBytes +
                               R::kEpiStagingBytes;
  // at least half the SM's shared memory, so that one CTA (which takes all of tensor
  // memory) runs per SM
  static constexpr int kSmemBytes = kUsed > 116 * 1024 ? kUsed : 116 * 1024;
  static_assert(kSmemBytes <= kSmemLimit, "resident weight does not fit");
};

struct TmParams {
  const __nv_bfloat16* feats;
  const int32_t* nbr;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  const __nv_bfloat16* residual;   // [N, O] or NULL (may equal out)
  int act;                         // subm3d_act
  int64_t N;
  int I, O;
  int ntiles;
  int* err;
  const int32_t* perm;             // tile plan: plan row -> output row, or NULL (identity)
  const uint32_t* tmask;           // tile plan: offsets present per tile, or NULL (all 27)
};

// Offsets a tile runs: its plan mask (the centre always included, so that every tile
// has a stage), or all 27 without a plan.
__device__ __forceinline__ uint32_t tm_tile_mask(const TmParams& p, int tile) {
  return p.tmask ? ((__ldg(p.tmask + tile) & 0x7FFFFFFu) | (1u << 13)) : 0x7FFFFFFu;
}
// The i-th (from 0) set bit of m: a binary search over popcounts of halves.
__device__ __forceinline__ int tm_nth_bit(uint32_t m, int i) {
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
// The offsets of pair j of a tile with mask m: its (2j)-th and (2j + 1)-th set bits
// (k1 = -1 when the pair has only one).
__device__ __forceinline__ void tm_pair_offsets(uint32_t m, int j, int& k0, int& k1) {
  k0 = tm_nth_bit(m, 2 * j);
  const uint32_t above = m & ~((2u << k0) - 1u);   // set bits after k0
  k1 = above ? __ffs(above) - 1 : -1;
}

__device__ __forceinline__ uint64_t tm_sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading offset (unused: swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

// kind::f16: fp32 accumulate, bf16 A and B, both K-major, M = 128.
template <int NMMA>
__device__ __forceinline__ uint32_t tm_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(NMMA >> 3) << 17) |
         (static_cast<uint32_t>(kBM >> 4) << 24);
}

__device__ __forceinline__ void tm_drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// One stage's MMAs with A in tensor memory: K step kk reads A columns a + 8 kk and
// the weight tile 32 bytes further (+2 in the descriptor's address field). Each MMA
// has its own operand registers; the first accumulates only if `acc` is set.
__device__ __forceinline__ void tm_mma_stage(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                             int ksteps, uint32_t acc) {
  const uint32_t a1 = a + 8, a2 = a + 16, a3 = a + 24;
  const uint64_t b1 = b + 2, b2 = b + 4, b3 = b + 6;
#define TM_MMA_HEAD                                                        \
  "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %9, 0;\n\t"                     \
  "elect.sync _|e, 0xffffffff;\n\t"                                        \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %10, p;\n\t"
#define TM_MMA(A, B) "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [" A "], " B ", %10, 1;\n\t"
#define TM_MMA_ARGS                                                                          \
  "r"(d), "r"(a), "r"(a1), "r"(a2), "r"(a3), "l"(b), "l"(b1), "l"(b2), "l"(b3), "r"(acc), \
      "r"(idesc)
  switch (ksteps) {
    case 4:
      asm volatile(TM_MMA_HEAD TM_MMA("%2", "%6") TM_MMA("%3", "%7") TM_MMA("%4", "%8") "}" ::TM_MMA_ARGS
                   : "memory");
      break;
    case 3:
      asm volatile(TM_MMA_HEAD TM_MMA("%2", "%6") TM_MMA("%3", "%7") "}" ::TM_MMA_ARGS : "memory");
      break;
    case 2:
      asm volatile(TM_MMA_HEAD TM_MMA("%2", "%6") "}" ::TM_MMA_ARGS : "memory");
      break;
    default:
      asm volatile(TM_MMA_HEAD "}" ::TM_MMA_ARGS : "memory");
      break;
  }
#undef TM_MMA_HEAD
#undef TM_MMA
#undef TM_MMA_ARGS
}

__device__ __forceinline__ void tm_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns from this thread's 32 registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


// 32 read-only bytes (8 words) from a 32-byte-aligned global address.
__device__ __forceinline__ void ld32B(const void* p, uint32_t* w) {
  asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

template <int NMMA, bool STAGED>
__global__ void __launch_bounds__(TmRoles<STAGED>::kThreads, 1)
    fwd_tm(const __grid_constant__ CUtensorMap wmap, const TmParams p) {
  using C = TmCfg<NMMA, STAGED>;
  using R = TmRoles<STAGED>;
  constexpr int kGroups = R::kGroups;
  constexpr int kStages = R::kStages;
  constexpr int kProducerWarps = R::kProducerWarps;
  constexpr int kMmaWarp = R::kMmaWarp;
  constexpr int kEpiWarp0 = R::kEpiWarp0;
  constexpr int kNbrWarp = R::kNbrWarp;
  constexpr int kWarpStaging = R::kWarpStaging;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sW = base;                                   // kStages slots of two taps
  const uint32_t sNbr = base + C::kWBytes;                    // 2 x 13.8 KB
  const int32_t* nbr_sm = reinterpret_cast<const int32_t*>(base_ptr + C::kWBytes);
  uint8_t* misc = base_ptr + C::kWBytes + 2 * kNbrTileBytes;
  // barriers: afull[12], aempty[12], accf[2], acce[2], nbrf[2], nbre[2], drain
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  const uint32_t afull0 = smem_u32(bars);
  const uint32_t aempty0 = afull0 + 8 * kStages;
  const uint32_t accf0 = aempty0 + 8 * kStages;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t nbrf0 = acce0 + 16;
  const uint32_t nbre0 = nbrf0 + 16;
  const uint32_t drain = nbre0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (2 * kStages + 9));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* bias_sm = reinterpret_cast<float*>(misc + 512);
  const uint32_t sStage = smem_u32(misc + 512 + 256 * 4);   // producers' row staging
  // epilogue row staging (per-thread form; there the producers' staging is empty)
  uint8_t* epi_stage = misc + 512 + 256 * 4 + R::kStagingBytes;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ntl = (p.ntiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                  static_cast<int>(gridDim.x);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(afull0 + 8 * s, 5);     // the group's four warps + the weight TMAs' expect_tx
      mbar_init(aempty0 + 8 * s, 1);    // one tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 128);
      mbar_init(nbrf0 + 8 * b, 1);
      mbar_init(nbre0 + 8 * b, kProducerWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&wmap);
  }
  if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    for (int o = tid - kEpiWarp0 * 32; o < NMMA; o += 128)
      bias_sm[o] = (p.bias && o < p.O) ? __bfloat162float(p.bias[o]) : 0.f;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------------ producers
    const int grp = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // row of the tile = tensor-memory lane
    const bool leader = quarter == 0 && lane == 0;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    bool bad = false, aborted = false;
    int cur = -1;                            // tile whose nbr block this warp is reading
    uint32_t last = 0;                       // one past the last stage this group issued
    // this thread's row of offset k of tile lt: its input row, -1 when absent
    auto row_index = [&](int lt, int k) -> int32_t {
      const int64_t row = int64_t(blockIdx.x + lt * gridDim.x) * kBM + r;
      if (row >= p.N) return -1;
      int32_t j = nbr_sm[(lt & 1) * (kBM * 27) + r * 27 + k];
      if (j < -1 || j >= p.N) {
        bad = true;
        j = -1;
      }
      return j;
    };
    // The warp's 32 rows of one offset are gathered with coalesced 16-byte copies (eight
    // lanes per row, four rows per instruction) into the warp's staging area, each row
    // 128 bytes with its 16-byte chunks rotated by (row & 7) so that neither the copies
    // nor the row reads below conflict; then every lane reads its own row back. Loading
    // whole rows per instruction costs the L1 data pipe one pass per 128-byte row
    // instead of one per 16 bytes of each lane's own row.
    // each lane's own row into registers: four 32-byte read-only loads (the form without
    // staging, for the dense offsets of input-order tiles)
    auto load_row = [&](int32_t j, uint32_t (&v)[32]) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {   // 16 channels (32 bytes) per load
        if (j >= 0 && q * 16 < p.I) {
          ld32B(p.feats + int64_t(j) * p.I + q * 16, v + 8 * q);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[8 * q + e] = 0u;
        }
      }
    };
    // buffer b of the warp holds the rows of the stage's offset b, so that both offsets'
    // copies are in flight at once
    const uint32_t stage_base = sStage + warp * kWarpStaging;
    auto gather_issue = [&](int32_t jown, int b) {   // jown: this lane's input row (-1: absent)
      const int c = lane & 7;
      const uint32_t buf = stage_base + b * kRowsStaging;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3);
        const int32_t j = __shfl_sync(0xffffffffu, jown, rr);
        if (j >= 0 && c * 8 < p.I)
          cp_async_16_ca(buf + rr * 128 + ((c ^ (rr & 7)) << 4),
                         p.feats + int64_t(j) * p.I + c * 8);
      }
      cp_async_commit();
    };
    // younger: copy groups issued after this one that may still be in flight (0 or 1)
    auto gather_finish = [&](int32_t jown, int b, int younger, uint32_t (&v)[32]) {
      if (younger) cp_async_wait_group1();
      else cp_async_wait_all();
      __syncwarp();
      const uint32_t buf = stage_base + b * kRowsStaging;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (jown >= 0 && c * 8 < p.I) q = ld_shared_v4(buf + lane * 128 + ((c ^ (lane & 7)) << 4));
        v[4 * c] = q.x;
        v[4 * c + 1] = q.y;
        v[4 * c + 2] = q.z;
        v[4 * c + 3] = q.w;
      }
      __syncwarp();   // every lane has its row: the staging area is free again
    };
    // Moves this warp's hold on the double-buffered nbr blocks forward to tile `to`,
    // taking part in every tile on the way (a tile with fewer stages than there are
    // groups has none for some groups): each tile's block is waited for, then released
    // when the next one is taken, so that every block's phases see all producer warps.
    auto advance_to = [&](int to) -> bool {
      for (int x = cur + 1; x <= to; ++x) {
        if (x > 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(nbre0 + 8 * ((x - 1) & 1));
        }
        const bool ok = mbar_wait(nbrf0 + 8 * (x & 1), (x >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) return false;
        cur = x;
      }
      return true;
    };
    // stage g of this CTA is pair g - g0 of local tile lt (whose pairs start at g0)
    int lt = 0;
    uint32_t g0 = 0, tm = ntl > 0 ? tm_tile_mask(p, blockIdx.x) : 1u;
    uint32_t np = (__popc(tm) + 1) / 2;
    for (uint32_t g = grp;; g += kGroups) {
      while (lt < ntl && g >= g0 + np) {
        g0 += np;
        ++lt;
        if (lt < ntl) {
          tm = tm_tile_mask(p, blockIdx.x + lt * gridDim.x);
          np = (__popc(tm) + 1) / 2;
        }
      }
      if (lt >= ntl) break;
      int k0, k1;
      tm_pair_offsets(tm, static_cast<int>(g - g0), k0, k1);
      const bool two = k1 >= 0;
      if (lt != cur && !advance_to(lt)) {
        aborted = true;
        break;
      }
      uint32_t v[32];
      const int32_t j0 = row_index(lt, k0);
      const int32_t j1 = two ? row_index(lt, k1) : -1;
      if constexpr (STAGED) {
        gather_issue(j0, 0);   // both offsets' rows in flight while the slot frees
        if (two) gather_issue(j1, 1);
      } else {
        load_row(j0, v);       // in flight while the slot frees
      }
      const uint32_t s = g % kStages;
      const uint32_t use = g / kStages;
      const bool ok = mbar_wait(aempty0 + 8 * s, (use & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        aborted = true;
        break;
      }
      if (leader) {   // the stage's weight taps into its slot
        mbar_arrive_expect_tx(afull0 + 8 * s, (two ? 2 : 1) * C::kTapBytes);
        tma_load_3d(sW + s * 2 * C::kTapBytes, &wmap, afull0 + 8 * s, 0, k0, 0);
        if (two) tma_load_3d(sW + (s * 2 + 1) * C::kTapBytes, &wmap, afull0 + 8 * s, 0, k1, 0);
      }
      last = g + kGroups;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_addr + kAColBase + s * kStageCols;
      if constexpr (STAGED) gather_finish(j0, 0, two ? 1 : 0, v);
      tmem_st32(taddr, v);
      if (two) {
        tmem_st_wait();   // v is free again
        if constexpr (STAGED) gather_finish(j1, 1, 0, v);
        else load_row(j1, v);
        tmem_st32(taddr + kOffCols, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(afull0 + 8 * s);
    }
    // the tiles after this group's last stage: taken and released like the others, so
    // that the loader warp can refill their buffers
    if (!aborted && cur < ntl - 1 && !advance_to(ntl - 1)) aborted = true;
    if (bad) atomicOr(p.err, kDevErrBadNbr);
    if (aborted && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, kDevErrTimeout);
    }
    if (aborted && leader) {   // no weight TMA of this group may still be landing
      for (uint32_t x = last >= static_cast<uint32_t>(kStages) ? last - kStages : 0u; x < last; ++x)
        if (x % kGroups == static_cast<uint32_t>(grp))
          tm_drain_wait(afull0 + 8 * (x % kStages), (x / kStages) & 1u);
    }
  } else if (warp == kNbrWarp) {
    // ------------------------------------------------------------------ nbr staging
    if (lane == 0) {
      int issued = 0;
      bool aborted = false;
      for (int lt = 0; lt < ntl; ++lt, ++issued) {
        const uint32_t nb = lt & 1;
        if (!mbar_wait(nbre0 + 8 * nb, ((lt >> 1) & 1) ^ 1, abort_flag)) {
          aborted = true;
          break;
        }
        const int64_t row0 = int64_t(blockIdx.x + lt * gridDim.x) * kBM;
        const int64_t rows = (p.N - row0) < kBM ? (p.N - row0) : kBM;
        const uint32_t bytes = static_cast<uint32_t>(rows) * 108u;
        const uint32_t bulk = bytes & ~15u;
        int32_t* dst = const_cast<int32_t*>(nbr_sm) + nb * (kBM * 27);
        for (uint32_t off = bulk; off < bytes; off += 4)   // ragged tail of the last tile
          dst[off / 4] = __ldg(p.nbr + row0 * 27 + off / 4);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(nbrf0 + 8 * nb, bulk);
        bulk_load(sNbr + nb * kNbrTileBytes, p.nbr + row0 * 27, bulk, nbrf0 + 8 * nb);
        if (lt + 2 < ntl) {   // the block after next into L2
          const int64_t row2 = int64_t(blockIdx.x + (lt + 2) * gridDim.x) * kBM;
          const int64_t rows2 = (p.N - row2) < kBM ? (p.N - row2) : kBM;
          const uint32_t b2 = static_cast<uint32_t>(rows2 * 108) & ~15u;
          if (b2) bulk_prefetch_l2(p.nbr + row2 * 27, b2);
        }
      }
      // every copy this warp issued has landed before the CTA may exit
      for (int x = issued > 2 ? issued - 2 : 0; x < issued; ++x)
        tm_drain_wait(nbrf0 + 8 * (x & 1), (x >> 1) & 1);
      if (aborted) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issue
    const uint32_t idesc = tm_idesc<NMMA>();
    const int ksteps = (p.I + 15) / 16;
    const uint64_t w0 = tm_sw128_desc(sW);
    bool aborted = false;
    uint32_t g = 0;
    for (int t = 0; t < ntl && !aborted; ++t) {
      const uint32_t buf = t & 1u;
      const uint32_t use = t >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(acce0 + 8 * buf, (use & 1u) ^ 1u, abort_flag))) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * kAccCols;
      const int noff = __popc(tm_tile_mask(p, blockIdx.x + t * gridDim.x));
      const int npairs = (noff + 1) / 2;
      for (int pr = 0; pr < npairs; ++pr, ++g) {
        const uint32_t s = g % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(afull0 + 8 * s, (g / kStages) & 1u, abort_flag))) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t a = tmem_base + kAColBase + s * kStageCols;
        const uint64_t b = w0 + static_cast<uint64_t>(2 * s) * (C::kTapBytes >> 4);
        tm_mma_stage(d_tmem, a, b, idesc, ksteps, pr == 0 ? 0u : 1u);
        if (2 * pr + 1 < noff)
          tm_mma_stage(d_tmem, a + kOffCols, b + (C::kTapBytes >> 4), idesc, ksteps, 1u);
        tm_commit(aempty0 + 8 * s);
      }
      if (!aborted) tm_commit(accf0 + 8 * buf);
    }
    if (aborted) {
      if (lane == 0) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
      tm_commit(drain);   // wait for every MMA already issued
      if (lane == 0) tm_drain_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int lg = warp & 3;                  // tensor-memory lane group of this warp
    uint8_t* stg = epi_stage + (warp - kEpiWarp0) * 32 * R::kEpiPitch;
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
      // (warp-uniform: the staged write-out below is a warp-wide step)
      const bool acc_ok = mbar_wait(accf0 + 8 * buf, use & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, acc_ok)) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + buf * kAccCols;
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
        if (row < p.N) {
          const uint4 y = epilogue8_bf16(v, bias_sm + col0, rrow != nullptr, rcur, p.act);
          if constexpr (STAGED) {
            // streaming store: the output is not read again here, the gathered rows are
            __stcs(reinterpret_cast<uint4*>(orow + col0), y);
          } else {   // into this lane's staging row (the pad makes the 32 rows conflict-free)
            *reinterpret_cast<uint4*>(stg + lane * R::kEpiPitch + cc * 16) = y;
          }
        }
      }
      if constexpr (!STAGED) {
        // the warp's 32 rows out of shared memory, whole rows per group of lanes (a row's
        // 16-byte pieces on consecutive lanes), each to the output row its lane named
        __syncwarp();
        constexpr int kPieces = NMMA / 8;   // 16-byte pieces per row (O = NMMA here)
        for (int e = lane; e < 32 * kPieces; e += 32) {
          const int rr = e / kPieces, c = e - rr * kPieces;
          const int64_t orr = __shfl_sync(0xffffffffu, row, rr);
          if (orr < p.N && c * 8 < p.O)
            __stcs(reinterpret_cast<uint4*>(p.out + orr * p.O) + c,
                   *reinterpret_cast<const uint4*>(stg + rr * R::kEpiPitch + c * 16));
        }
        __syncwarp();   // the staging rows are free for the next tile
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, 512);
}

typedef CUresult (*TmEncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

TmEncodeTiledFn tm_get_encode() {
  static TmEncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TmEncodeTiledFn>(f);
  });
  return fn;
}

template <int NMMA, bool STAGED>
int tm_launch(const TmParams& prm, const __nv_bfloat16* weight, cudaStream_t stream) {
  using C = TmCfg<NMMA, STAGED>;
  static PerDevice<bool> attr_set;
  const int arc = set_smem_limit_once(attr_set,
                                      reinterpret_cast<const void*>(fwd_tm<NMMA, STAGED>),
                                      C::kSmemBytes, "fwd_tm");
  if (arc != SUBM3D_OK) return arc;
  TmEncodeTiledFn encode = tm_get_encode();
  if (!encode) {
    set_error("subm3d_forward: cuTensorMapEncodeTiled is not available from the driver");
    return SUBM3D_ERR_CUDA;
  }
  // weight [O, 3, 3, 3, I] as a 3-D tensor {I, 27, O}; box = one tap's [O x 64] slice
  CUtensorMap wmap;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(prm.I), 27, static_cast<cuuint64_t>(prm.O)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(prm.I) * 2,
                                 static_cast<cuuint64_t>(prm.I) * 27 * 2};
  const cuuint32_t box[3] = {64, 1, NMMA};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                            const_cast<__nv_bfloat16*>(weight), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("subm3d_forward: cuTensorMapEncodeTiled failed (%d) for weight=%p I=%d O=%d",
              static_cast<int>(r), (const void*)weight, prm.I, prm.O);
    return SUBM3D_ERR_CUDA;
  }
  const int grid = prm.ntiles < num_sms() ? prm.ntiles : num_sms();
  fwd_tm<NMMA, STAGED><<<grid, TmRoles<STAGED>::kThreads, C::kSmemBytes, stream>>>(wmap, prm);
  SUBM3D_LAUNCHED("fwd_tm");
  return SUBM3D_OK;
}

}  // namespace

bool forward_tm_applies(const void* feats, int I, int O) {
  (void)feats;   // 16-byte alignment, checked for every call, is all the copies need
  return I >= 16 && I <= 64 && I % 16 == 0 && O >= 16 && O <= 64 && O % 16 == 0;
}

int forward_launch_tm(const __nv_bfloat16* feats, const int32_t* nbr, const __nv_bfloat16* weight,
                      const __nv_bfloat16* bias, __nv_bfloat16* out, int64_t N, int I, int O,
                      Epilogue epi, TilePlan plan, cudaStream_t stream) {
  const int64_t ntiles = (N + kBM - 1) / kBM;
  if (ntiles > 0x7FFFFFFFll) {
    set_error("subm3d_forward: N=%lld too large", (long long)N);
    return SUBM3D_ERR_UNSUPPORTED;
  }
  int* err = forward_error_word();
  if (!err) return SUBM3D_ERR_CUDA;
  TmParams prm{feats, nbr, bias, out, static_cast<const __nv_bfloat16*>(epi.residual),
               epi.act, N, I, O, static_cast<int>(ntiles), err, plan.perm, plan.tmask};
  // Tiles of a mask-grouped plan run about half the offsets, so their fewer stages can
  // afford whole-row copies through shared memory (which spare the L1 data pipe); dense
  // tiles (input order, or a plan of small windows such as the Morton order) run most
  // offsets and go faster with each lane loading its own row, which needs 32-byte-
  // aligned rows.
  const bool staged = (plan.tmask != nullptr && !plan.dense) ||
                      (reinterpret_cast<uintptr_t>(feats) & 31) != 0;
  switch (O) {
    case 16: return staged ? tm_launch<16, true>(prm, weight, stream)
                           : tm_launch<16, false>(prm, weight, stream);
    case 32: return staged ? tm_launch<32, true>(prm, weight, stream)
                           : tm_launch<32, false>(prm, weight, stream);
    case 48: return staged ? tm_launch<48, true>(prm, weight, stream)
                           : tm_launch<48, false>(prm, weight, stream);
    case 64: return staged ? tm_launch<64, true>(prm, weight, stream)
                           : tm_launch<64, false>(prm, weight, stream);
    default:
      set_error("subm3d_forward: O=%d outside the narrow tensor-core kernel's range", O);
      return SUBM3D_ERR_UNSUPPORTED;
  }
}

}  // namespace subm3d
