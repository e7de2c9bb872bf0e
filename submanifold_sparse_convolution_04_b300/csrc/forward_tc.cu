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
//   A = the 128 gathered neighbour rows, 64 channels each (16 KB), staged by 128
//       producer threads with 16-byte cp.async (an absent neighbour, nbr = -1,
//       zero-fills and reads nothing), written in the 128-byte-swizzled K-major
//       layout the tensor core reads. Each producer marks the stage full with
//       cp.async.mbarrier.arrive.noinc, so a slot counts as full the moment its
//       rows land and no producer ever blocks on its own copies; the MMA thread
//       orders those generic-proxy writes before its tensor-core reads with
//       fence.proxy.async after the barrier wait;
//   B = W_k[:, chunk] = weight[:, kz, ky, kx, chunk], an [O x 64] K-major tile (I is
//       contiguous in the checkpoint layout, so no transpose), fetched by TMA with
//       the same 128-byte swizzle; out-of-range rows/columns are zero-filled.
// One thread issues tcgen05.mma (M = 128, N = round_up(O, 16), K = 16 per
// instruction) into a tensor-memory accumulator; tcgen05.commit frees the stage.
// Two accumulators (double-buffered tensor memory) let four epilogue warps drain
// tile t (tcgen05.ld -> + bias -> bf16 round-to-nearest-even -> one store per
// element) while the tensor core works on tile t + 1.
//
// Warp roles (320 threads): warps 0-3 producers (thread 0 also issues the weight
// TMA), warp 4 tensor-memory allocation + MMA issue (one lane), warps 5-8 epilogue,
// warp 9 stages each tile's 128 x 27 block of nbr (13.8 KB, contiguous in memory)
// into a double-buffered shared-memory ring with one bulk async copy, a tile
// ahead, so the producers never wait on a global load before issuing a gather.
// Every mbarrier wait is bounded (kWaitLimitNs); a wait that runs out sets the
// device error word, stops the CTA's pipeline, drains what is in flight and
// releases tensor memory before the CTA exits.
#include <mutex>

#include "common.cuh"

namespace subm3d {

__device__ int g_forward_err;

int* forward_error_word() {
  static int* ptr = nullptr;
  if (!ptr) cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_forward_err);
  return ptr;
}

namespace {

constexpr int kBM = 128;          // output rows per tile (tensor-memory lanes)
constexpr int kKC = 64;           // channels per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 320;
constexpr int kProducerThreads = 128;
constexpr int kMmaWarp = 4;
constexpr int kNbrWarp = 9;
constexpr int kNbrTileBytes = kBM * 27 * 4;   // one tile's rows of nbr
constexpr int kSmemLimit = 227 * 1024;

template <int NMMA>
struct Cfg {
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = NMMA * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kMisc = 1024 /*alignment slack*/ + 2 * kNbrTileBytes /*nbr ring*/ +
                               512 /*barriers*/ + 4 * 256 /*bias*/;
  static constexpr int kFit = (kSmemLimit - kMisc) / kStageBytes;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;
  static constexpr int kTmemCols = (2 * NMMA <= 32) ? 32 : (2 * NMMA <= 64) ? 64
                                 : (2 * NMMA <= 128) ? 128 : (2 * NMMA <= 256) ? 256 : 512;
  static constexpr int kSmemBytes = kMisc + kStages * kStageBytes;
  static_assert(kStages >= 3, "pipeline too shallow");
};

struct Params {
  const __nv_bfloat16* feats;
  const int32_t* nbr;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  int64_t N;
  int I, O;
  int nchunks;
  int ntiles;
  int* err;
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

template <int NMMA>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc(const __grid_constant__ CUtensorMap wmap, const Params p) {
  using C = Cfg<NMMA>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base;                              // S x 16 KB
  const uint32_t sB = base + S * C::kABytes;             // S x NMMA*128 B
  const uint32_t sNbr = base + S * C::kStageBytes;       // 2 x 13.8 KB
  const int32_t* nbr_sm = reinterpret_cast<const int32_t*>(base_ptr + S * C::kStageBytes);
  uint8_t* misc = base_ptr + S * C::kStageBytes + 2 * kNbrTileBytes;
  // barriers: full[S], empty[S], accf[2], acce[2], drain, nbrf[2], nbre[2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t accf0 = empty0 + 8 * S;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  const uint32_t nbrf0 = drain + 8;
  const uint32_t nbre0 = nbrf0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (2 * S + 9));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* bias_sm = reinterpret_cast<float*>(misc + 512);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, kProducerThreads + 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 128);
      mbar_init(nbrf0 + 8 * b, 1);
      mbar_init(nbre0 + 8 * b, kProducerThreads);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&wmap);
  }
  if (tid >= 160 && tid < 288) {
    for (int o = tid - 160; o < NMMA; o += 128)
      bias_sm[o] = (p.bias && o < p.O) ? __bfloat162float(p.bias[o]) : 0.f;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------------ producers
    const int q = tid & 7;          // 16-byte column chunk inside the 128-byte row
    const int rsub = tid >> 3;      // rows rsub + 16 m, m = 0..7
    uint32_t g = 0, lt = 0;
    bool bad = false, aborted = false;
    for (int tile = blockIdx.x; tile < p.ntiles && !aborted; tile += gridDim.x, ++lt) {
      const int64_t row0 = int64_t(tile) * kBM;
      const uint32_t nb = lt & 1u;
      if (!mbar_wait(nbrf0 + 8 * nb, (lt >> 1) & 1u, abort_flag)) {
        aborted = true;
        break;
      }
      const int32_t* tile_nbr = nbr_sm + nb * (kBM * 27);
      for (int k = 0; k < 27 && !aborted; ++k) {
        int32_t j[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int r = rsub + 16 * m;
          int32_t v = -1;
          if (row0 + r < p.N) {
            v = tile_nbr[r * 27 + k];
            if (v < -1 || v >= p.N) {
              bad = true;
              v = -1;
            }
          }
          j[m] = v;
        }
        if (k == 26) mbar_arrive(nbre0 + 8 * nb);   // this tile's nbr block is no longer read
        for (int c = 0; c < p.nchunks; ++c) {
          const uint32_t s = g % S;
          const uint32_t ph = (g / S) & 1u;
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) {
            aborted = true;
            break;
          }
          if (tid == 0) {
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
          ++g;
        }
      }
    }
    cp_async_wait_all();   // no gather of this thread is still landing when the CTA exits
    if (bad) atomicOr(p.err, kDevErrBadNbr);
    if (aborted) {
      *abort_flag = 1;
      atomicOr(p.err, kDevErrTimeout);
      if (tid == 0) {   // make sure no TMA write is still landing in this CTA's memory
        for (uint32_t x = (g > static_cast<uint32_t>(S) ? g - S : 0u); x < g; ++x)
          drain_wait(full0 + 8 * (x % S), (x / S) & 1u);
      }
    }
  } else if (warp == kNbrWarp) {
    // ------------------------------------------------------------------ nbr staging
    if (lane == 0) {
      uint32_t lt = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++lt) {
        const uint32_t nb = lt & 1u;
        if (!mbar_wait(nbre0 + 8 * nb, ((lt >> 1) & 1u) ^ 1u, abort_flag)) {
          aborted = true;
          break;
        }
        const int64_t row0 = int64_t(tile) * kBM;
        const int64_t rows = (p.N - row0) < kBM ? (p.N - row0) : kBM;
        const uint32_t bytes = static_cast<uint32_t>(rows) * 108u;
        const uint32_t bulk = bytes & ~15u;
        int32_t* dst = const_cast<int32_t*>(nbr_sm) + nb * (kBM * 27);
        for (uint32_t off = bulk; off < bytes; off += 4)   // ragged tail of the last tile
          dst[off / 4] = __ldg(p.nbr + row0 * 27 + off / 4);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(nbrf0 + 8 * nb, bulk);
        bulk_load(sNbr + nb * kNbrTileBytes, p.nbr + row0 * 27, bulk, nbrf0 + 8 * nb);
      }
      // every copy this warp issued has landed before the CTA may exit
      const uint32_t issued = lt;
      for (uint32_t x = issued > 2 ? issued - 2 : 0; x < issued; ++x)
        drain_wait(nbrf0 + 8 * (x & 1u), (x >> 1) & 1u);
      if (aborted) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = make_idesc<NMMA>();
      uint32_t g = 0, t = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < p.ntiles && !aborted; tile += gridDim.x, ++t) {
        const uint32_t buf = t & 1u;
        const uint32_t use = t >> 1;
        if (!mbar_wait(acce0 + 8 * buf, (use & 1u) ^ 1u, abort_flag)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * NMMA;
        uint32_t accumulate = 0;
        for (int k = 0; k < 27 && !aborted; ++k) {
          for (int c = 0; c < p.nchunks; ++c) {
            const uint32_t s = g % S;
            const uint32_t ph = (g / S) & 1u;
            if (!mbar_wait(full0 + 8 * s, ph, abort_flag)) {
              aborted = true;
              break;
            }
            fence_proxy_async_smem();
            tc_fence_after();
            const int rem = p.I - c * kKC;
            const int ksteps = rem >= kKC ? 4 : (rem + 15) / 16;
            const uint32_t a0 = sA + s * C::kABytes;
            const uint32_t b0 = sB + s * C::kBBytes;
            for (int kk = 0; kk < ksteps; ++kk) {
              tc_mma_f16(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                         accumulate);
              accumulate = 1;
            }
            tc_commit(empty0 + 8 * s);
            ++g;
          }
        }
        if (!aborted) tc_commit(accf0 + 8 * buf);
      }
      if (aborted) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
        tc_commit(drain);            // wait for every MMA already issued
        drain_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int lg = warp & 3;                  // tensor-memory lane group of this warp
    uint32_t t = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++t) {
      const uint32_t buf = t & 1u;
      const uint32_t use = t >> 1;
      if (!mbar_wait(accf0 + 8 * buf, use & 1u, abort_flag)) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
        break;
      }
      tc_fence_after();
      const int64_t row = int64_t(tile) * kBM + lg * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + buf * NMMA;
      __nv_bfloat16* orow = p.out + row * p.O;
#pragma unroll 1
      for (int cc = 0; cc < NMMA / 16; ++cc) {
        uint32_t v[16];
        tmem_ld16(taddr + cc * 16, v);
        tmem_ld_wait();
        if (cc == NMMA / 16 - 1) {
          tc_fence_before();
          mbar_arrive(acce0 + 8 * buf);
        }
        const int col0 = cc * 16;
        if (row < p.N && col0 < p.O) {
          uint32_t packed[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float lo = __uint_as_float(v[2 * e]) + bias_sm[col0 + 2 * e];
            const float hi = __uint_as_float(v[2 * e + 1]) + bias_sm[col0 + 2 * e + 1];
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
            packed[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + col0);
          dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          if (col0 + 8 < p.O) dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
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

template <int NMMA>
int launch(const Params& prm, const __nv_bfloat16* weight, cudaStream_t stream) {
  using C = Cfg<NMMA>;
  static bool attr_set = false;
  if (!attr_set) {
    SUBM3D_CUDA_TRY(cudaFuncSetAttribute(fwd_tc<NMMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes));
    attr_set = true;
  }
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
  const int grid = prm.ntiles < num_sms() ? prm.ntiles : num_sms();
  fwd_tc<NMMA><<<grid, kThreads, C::kSmemBytes, stream>>>(map, prm);
  SUBM3D_LAUNCHED("fwd_tc");
  return SUBM3D_OK;
}

}  // namespace

int forward_launch_tc(const __nv_bfloat16* feats, const int32_t* nbr, const __nv_bfloat16* weight,
                      const __nv_bfloat16* bias, __nv_bfloat16* out, int64_t N, int I, int O,
                      cudaStream_t stream) {
  const int64_t ntiles = (N + kBM - 1) / kBM;
  if (ntiles > 0x7FFFFFFFll) {
    set_error("subm3d_forward: N=%lld too large", (long long)N);
    return SUBM3D_ERR_UNSUPPORTED;
  }
  Params prm{feats, nbr, bias, out, N, I, O, (I + kKC - 1) / kKC, static_cast<int>(ntiles),
             forward_error_word()};
  const int nmma = (O + 15) / 16 * 16;
  switch (nmma) {
#define SUBM3D_CASE(n) \
  case n:              \
    return launch<n>(prm, weight, stream);
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
