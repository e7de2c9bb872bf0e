// Internal helpers shared by the libsubm3d.so translation units: status and message
// plumbing, the kernel-launch counter, and thin inline-PTX wrappers for the sm_103a
// features the kernels use (mbarrier, cp.async, TMA bulk tensor copies, tcgen05).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/subm3d.h"

namespace subm3d {

// ---------------------------------------------------------------------------- host side

void set_error(const char* fmt, ...);          // thread-local message, printf-style
void clear_error();
void count_launch(int n = 1);                  // host-side kernel-launch counter

// Checks a CUDA runtime return code; on failure records the message and returns
// SUBM3D_ERR_CUDA from the enclosing function.
#define SUBM3D_CUDA_TRY(expr)                                                          \
  do {                                                                                 \
    cudaError_t e_ = (expr);                                                           \
    if (e_ != cudaSuccess) {                                                           \
      ::subm3d::set_error("%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_),     \
                          __FILE__, __LINE__);                                         \
      return SUBM3D_ERR_CUDA;                                                          \
    }                                                                                  \
  } while (0)

// After a kernel launch: counts it and turns a launch error into SUBM3D_ERR_CUDA.
#define SUBM3D_LAUNCHED(name)                                                          \
  do {                                                                                 \
    ::subm3d::count_launch();                                                          \
    cudaError_t e_ = cudaGetLastError();                                               \
    if (e_ != cudaSuccess) {                                                           \
      ::subm3d::set_error("launch of %s failed: %s", name, cudaGetErrorString(e_));   \
      return SUBM3D_ERR_CUDA;                                                          \
    }                                                                                  \
  } while (0)

// Host state that belongs to one device (kernel attributes, symbol addresses, SM
// counts) is kept per device ordinal, filled on the first call made with that device
// current, under a mutex, so that calls on several devices or from several threads
// each see their own device's values.
constexpr int kMaxDevices = 64;

// The current device in *dev; SUBM3D_ERR_CUDA or SUBM3D_ERR_UNSUPPORTED (ordinal
// outside [0, kMaxDevices)) with the message set otherwise.
int current_device(int* dev);

template <typename T>
class PerDevice {
 public:
  // The value for the current device in *out, made by make(T*) -> status on that
  // device's first call (a failed make is retried on the next call).
  template <typename F>
  int get(T* out, F&& make) {
    int dev = 0;
    const int rc = current_device(&dev);
    if (rc != SUBM3D_OK) return rc;
    std::lock_guard<std::mutex> lock(mu_);
    if (!ready_[dev]) {
      const int mrc = make(&val_[dev]);
      if (mrc != SUBM3D_OK) return mrc;
      ready_[dev] = true;
    }
    *out = val_[dev];
    return SUBM3D_OK;
  }

 private:
  std::mutex mu_;
  bool ready_[kMaxDevices] = {};
  T val_[kMaxDevices] = {};
};

// SM count of the current device (148 if it cannot be read: only grid sizes depend on it).
int num_sms();

// Sets a kernel's dynamic shared-memory limit once per device.
int set_smem_limit_once(PerDevice<bool>& done, const void* kernel, int bytes, const char* name);

// Device error word of the forward, upsample and pixel-shuffle kernels and of the
// asynchronous kernel-map builds (bit flags below).
enum : int {
  kDevErrBadNbr = 1, kDevErrTimeout = 2, kDevErrBadParent = 4, kDevErrKmapCoord = 8,
  kDevErrKmapDup = 16, kDevErrKmapFull = 32, kDevErrKmapInternal = 64, kDevErrBadPlan = 128,
  kDevErrBadOrder = 256   // an asynchronous downsample given an order that is not Morton order
};

// Tile plan (subm3d_build_kmap_grouped): the caller's buffer holds, 256-byte aligned,
//   perm      int32 [N]       plan row -> input row
//   nbr       int32 [N, 27]   row r: the neighbour table row of input row perm[r]
//   tile_mask uint32 [ntiles] tile t (plan rows 128 t .. 128 t + 127): bit k set when
//                             some row of the tile has a neighbour at offset k
constexpr int kPlanTileRows = 128;
struct PlanLayout {
  size_t perm, nbr, tmask, total;
  int64_t ntiles;
};
inline PlanLayout plan_layout(int64_t N) {
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  PlanLayout P;
  P.ntiles = (N + kPlanTileRows - 1) / kPlanTileRows;
  size_t o = 0;
  P.perm = o;  o = a256(o + sizeof(int32_t) * N);
  P.nbr = o;   o = a256(o + sizeof(int32_t) * 27 * N);
  P.tmask = o; o = a256(o + sizeof(uint32_t) * P.ntiles);
  P.total = o;
  return P;
}
// What the forward kernels read of a plan: perm and tile_mask NULL for the plain
// (input-order, all offsets) path.
struct TilePlan {
  const int32_t* perm;
  const uint32_t* tmask;
  // a plan whose tiles keep most of their offsets (windows below 4096 voxels, the Morton
  // order at window 1): the narrow kernel then loads rows per thread, as without a plan
  bool dense = false;
};
// Device address of the word on the current device, or NULL (message set) when it
// cannot be had; a launcher then returns SUBM3D_ERR_CUDA without launching.
int* forward_error_word();
// Fused epilogue of subm3d_forward_ex: out = act(acc + bias + residual); residual NULL
// and act SUBM3D_ACT_NONE give the plain convolution.
struct Epilogue {
  const void* residual;   // [N, O] of the feature dtype, or NULL
  int act;                // subm3d_act
};
int forward_launch_tc(const __nv_bfloat16* feats, const int32_t* nbr,
                      const __nv_bfloat16* weight, const __nv_bfloat16* bias,
                      __nv_bfloat16* out, int64_t N, int I, int O, Epilogue epi,
                      TilePlan plan, cudaStream_t stream);
// The narrow-layer kernel (A operand in tensor memory): I and O in {16, 32, 48, 64}.
bool forward_tm_applies(const void* feats, int I, int O);
int forward_launch_tm(const __nv_bfloat16* feats, const int32_t* nbr,
                      const __nv_bfloat16* weight, const __nv_bfloat16* bias,
                      __nv_bfloat16* out, int64_t N, int I, int O, Epilogue epi,
                      TilePlan plan, cudaStream_t stream);
int forward_launch_simt(const void* feats, const int32_t* nbr, const void* weight,
                        const void* bias, void* out, int64_t N, int I, int O,
                        subm3d_dtype dtype, Epilogue epi, TilePlan plan, cudaStream_t stream);
int kmap_build(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr, int32_t* order,
               int64_t hash_capacity, void* workspace, size_t ws_bytes, cudaStream_t stream);
int kmap_build_async(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                     void* workspace, size_t ws_bytes, cudaStream_t stream);
size_t kmap_grouped_workspace_bytes(int64_t N);
void kmap_stage_timing(bool on);
int kmap_stage_times(float* ms, const char** names, int max);
int kmap_build_grouped(const int32_t* coords, int64_t N, int32_t res, int64_t window, void* plan,
                       size_t plan_bytes, void* workspace, size_t ws_bytes, bool sync,
                       cudaStream_t stream);
size_t kmap_workspace_bytes(int64_t N, int64_t hash_capacity);
size_t downsample_workspace_bytes(int64_t N);
int downsample_build(const int32_t* coords, int64_t N, int32_t res, const int32_t* order,
                     const void* feats, int32_t C, subm3d_dtype dtype, int mode,
                     int32_t* coarse_coords, void* coarse_feats, int32_t* parent,
                     uint8_t* child_mask, int64_t* M_out, void* workspace, size_t ws_bytes,
                     cudaStream_t stream, int64_t* M_dev = nullptr);
int upsample_launch(const void* coarse_feats, int64_t M, int32_t C, const int32_t* parent,
                    int64_t N, subm3d_dtype dtype, void* fine_feats, cudaStream_t stream);
int spatial2channel_launch(const void* feats, const int32_t* coords, const int32_t* parent,
                           const uint8_t* child_mask, int64_t N, int64_t M, int32_t C,
                           subm3d_dtype dtype, void* out, cudaStream_t stream);
int channel2spatial_launch(const void* coarse_feats, const int32_t* coords, const int32_t* parent,
                           int64_t N, int64_t M, int32_t C, subm3d_dtype dtype, void* fine_feats,
                           cudaStream_t stream);
int64_t default_hash_capacity(int64_t N);

// ---------------------------------------------------------------------------- device side

// Limit of every bounded wait in the kernels (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// mbarrier -------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of parity `parity` to complete. Bounded: gives up after
// kWaitLimitNs, or as soon as *abort is set by another thread of the CTA; returns
// false in both cases (the caller then stops issuing work).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// cp.async (16 bytes; src_bytes = 0 writes zeros and reads nothing) ----------------
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// 16 bytes global -> shared, cached in L1 as well (rows that neighbouring voxels share
// are often read again soon).
__device__ __forceinline__ void cp_async_16_ca(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most one of this thread's committed cp.async groups is still pending.
__device__ __forceinline__ void cp_async_wait_group1() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Arrives on `bar` (counted in its expected count) once every cp.async this thread
// issued so far has landed in shared memory; the thread itself does not wait.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA ------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// Untiled bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16),
// completing on `bar` by transaction bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Untiled bulk copy shared -> global (16-byte aligned addresses, size a multiple of 16),
// tracked by this thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's bulk stores have read their shared-memory sources (which may be reused).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Asks the memory system to bring `bytes` at `src` into L2 (a hint: no completion, no
// effect on correctness). `src` 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// tcgen05 --------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives once on `bar` when every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// 32 lanes x 32 bit, 8 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Fused epilogue ------------------------------------------------------------------
// silu(y) = y / (1 + e^-y) with the fast exponential and division intrinsics (a few
// ulp, far below the bf16 output rounding and the fp32 tolerance; the exact expf and
// IEEE division made the epilogue warps, not the gathers, set the pace). Below -80,
// |silu(y)| < 1e-33 is returned as 0 (e^80 stays inside the intrinsic division's
// range); NaN propagates.
__device__ __forceinline__ float apply_act(float y, int act) {
  if (act == SUBM3D_ACT_RELU) return fmaxf(y, 0.f);
  if (act == SUBM3D_ACT_SILU) return y < -80.f ? 0.f : __fdividef(y, 1.f + __expf(-y));
  return y;
}
// silu(y) for an output that is rounded to bf16 next: y * sigmoid(y) with
// sigmoid(y) = (1 + tanh(y / 2)) / 2, tanh from the hardware approximation (relative
// error about 2^-11, below half a bf16 unit in the last place, 2^-9). One special-
// function instruction instead of an exponential and a division: the four epilogue
// warps, not the gathers, set the pace with the exact form.
__device__ __forceinline__ float silu_for_bf16(float y) {
  float t;
  const float h = 0.5f * y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}
// Asks L2 for every 128-byte line of a row of `bytes` (> 0) bytes at p; the addresses
// must lie inside the allocation. A hint: no data comes back, nothing waits for it.
__device__ __forceinline__ void prefetch_row_l2(const void* p, int bytes) {
  const char* c = static_cast<const char*>(p);
  for (int off = 0; off < bytes; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(c + bytes - 1));
}
// 16 bytes of a row that may be the output buffer itself (an in-place residual): a
// plain load, not the read-only path.
__device__ __forceinline__ uint4 ld_row16(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint4*>(p);
}
// Eight consecutive output columns of one row: acc (fp32 bit patterns) + bias, plus the
// eight residual values in r when has_res, then the activation, rounded to bf16
// (nearest-even) and packed for one 16-byte store.
__device__ __forceinline__ uint4 epilogue8_bf16(const uint32_t (&acc)[8], const float* bias8,
                                                bool has_res, uint4 r, int act) {
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = __uint_as_float(acc[e]) + bias8[e];
  if (has_res) {
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rw[e]));
      y[2 * e] += f.x;
      y[2 * e + 1] += f.y;
    }
  }
  if (act == SUBM3D_ACT_RELU) {
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = fmaxf(y[e], 0.f);
  } else if (act == SUBM3D_ACT_SILU) {
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = silu_for_bf16(y[e]);
  }
  uint32_t packed[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
    packed[e] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

}  // namespace subm3d
