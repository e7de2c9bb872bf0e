// C-ABI entry points of libsubm3d.so (declared in include/subm3d.h): host-side
// argument checks, the thread-local error message, the launch counter, and
// dispatch to the kernel-map and forward launchers.
#include <cstdarg>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace subm3d {

namespace {
thread_local char g_msg[512] = "";
std::atomic<int64_t> g_launches{0};
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}
void clear_error() { g_msg[0] = '\0'; }
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int current_device(int* dev) {
  *dev = -1;
  SUBM3D_CUDA_TRY(cudaGetDevice(dev));
  if (*dev < 0 || *dev >= kMaxDevices) {
    set_error("device ordinal %d outside [0, %d)", *dev, kMaxDevices);
    return SUBM3D_ERR_UNSUPPORTED;
  }
  return SUBM3D_OK;
}

namespace {
PerDevice<int> g_sms;
PerDevice<int*> g_err_word;
}  // namespace

int num_sms() {
  int sms = 0;
  const int rc = g_sms.get(&sms, [](int* v) -> int {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    *v = n;
    return static_cast<int>(SUBM3D_OK);
  });
  return rc == SUBM3D_OK ? sms : 148;
}

int set_smem_limit_once(PerDevice<bool>& done, const void* kernel, int bytes, const char* name) {
  bool ok = false;
  return done.get(&ok, [&](bool* v) -> int {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
      set_error("cudaFuncSetAttribute(%s, %d bytes of shared memory) failed: %s", name, bytes,
                cudaGetErrorString(e));
      return static_cast<int>(SUBM3D_ERR_CUDA);
    }
    *v = true;
    return static_cast<int>(SUBM3D_OK);
  });
}

// The device error word (kDevErr* bits) that the forward, upsample and pixel-shuffle
// kernels report into; one per device that loads the library.
__device__ int g_forward_err;

int* forward_error_word() {
  int* p = nullptr;
  const int rc = g_err_word.get(&p, [](int** v) -> int {
    void* a = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&a, g_forward_err);
    if (e != cudaSuccess || !a) {
      set_error("cudaGetSymbolAddress(device error word) failed: %s", cudaGetErrorString(e));
      return static_cast<int>(SUBM3D_ERR_CUDA);
    }
    *v = static_cast<int*>(a);
    return static_cast<int>(SUBM3D_OK);
  });
  return rc == SUBM3D_OK ? p : nullptr;
}

}  // namespace subm3d

using namespace subm3d;

extern "C" {

size_t subm3d_kmap_workspace_bytes(int64_t N) { return kmap_workspace_bytes(N, 0); }

size_t subm3d_kmap_workspace_bytes_ex(int64_t N, int64_t hash_capacity) {
  if (hash_capacity < 0) return 0;
  return kmap_workspace_bytes(N, hash_capacity);
}

int subm3d_build_kmap(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  clear_error();
  return kmap_build(coords, N, res, nbr, nullptr, 0, workspace, ws_bytes, stream);
}

int subm3d_build_kmap_ex(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                         int32_t* order, int64_t hash_capacity, void* workspace, size_t ws_bytes,
                         cudaStream_t stream) {
  clear_error();
  return kmap_build(coords, N, res, nbr, order, hash_capacity, workspace, ws_bytes, stream);
}

namespace {
// Host-side checks and kernel choice shared by the plain and the tile-plan forward.
int forward_dispatch(const char* fn, const void* feats, const int32_t* nbr, const void* weight,
                     const void* bias, const void* residual, subm3d_act act, void* out, int64_t N,
                     int32_t I, int32_t O, subm3d_dtype dtype, TilePlan plan,
                     cudaStream_t stream) {
  if (N < 0 || N > 0x7FFFFFFFll) {
    set_error("%s: N=%lld outside [0, 2^31)", fn, (long long)N);
    return SUBM3D_ERR_ARG;
  }
  if (I < 1 || I > 4096 || O < 1 || O > 4096) {
    set_error("%s: I=%d, O=%d must lie in [1, 4096]", fn, I, O);
    return SUBM3D_ERR_ARG;
  }
  if (dtype != SUBM3D_F32 && dtype != SUBM3D_BF16) {
    set_error("%s: unknown dtype %d", fn, static_cast<int>(dtype));
    return SUBM3D_ERR_ARG;
  }
  if (act != SUBM3D_ACT_NONE && act != SUBM3D_ACT_RELU && act != SUBM3D_ACT_SILU) {
    set_error("%s: unknown activation %d", fn, static_cast<int>(act));
    return SUBM3D_ERR_ARG;
  }
  if (N == 0) return SUBM3D_OK;
  if (!feats || !nbr || !weight || !out) {
    set_error("%s: NULL pointer (feats=%p nbr=%p weight=%p out=%p)", fn, feats,
              (const void*)nbr, weight, out);
    return SUBM3D_ERR_ARG;
  }
  const uintptr_t any = reinterpret_cast<uintptr_t>(feats) | reinterpret_cast<uintptr_t>(nbr) |
                        reinterpret_cast<uintptr_t>(weight) | reinterpret_cast<uintptr_t>(out) |
                        reinterpret_cast<uintptr_t>(bias) | reinterpret_cast<uintptr_t>(residual);
  if (any & 15) {
    set_error("%s: feats=%p nbr=%p weight=%p bias=%p residual=%p out=%p must be 16-byte aligned",
              fn, feats, (const void*)nbr, weight, bias, residual, out);
    return SUBM3D_ERR_ARG;
  }
  if (residual && residual != out) {
    // the one overlap allowed is residual == out (in place)
    const size_t bytes = static_cast<size_t>(N) * O * (dtype == SUBM3D_BF16 ? 2 : 4);
    const char* r = static_cast<const char*>(residual);
    const char* q = static_cast<const char*>(out);
    if (r < q + bytes && q < r + bytes) {
      set_error("%s: residual=%p partially overlaps out=%p (only residual == out is allowed)", fn,
                residual, out);
      return SUBM3D_ERR_ARG;
    }
  }
  const Epilogue epi{residual, static_cast<int>(act)};
  if (dtype == SUBM3D_BF16) {
    if (I % 8 || O % 8) {
      set_error("%s: bf16 needs I %% 8 == 0 and O %% 8 == 0 (got I=%d, O=%d)", fn, I, O);
      return SUBM3D_ERR_UNSUPPORTED;
    }
    if (forward_tm_applies(feats, I, O))
      return forward_launch_tm(static_cast<const __nv_bfloat16*>(feats), nbr,
                               static_cast<const __nv_bfloat16*>(weight),
                               static_cast<const __nv_bfloat16*>(bias),
                               static_cast<__nv_bfloat16*>(out), N, I, O, epi, plan, stream);
    if (O <= 256)
      return forward_launch_tc(static_cast<const __nv_bfloat16*>(feats), nbr,
                               static_cast<const __nv_bfloat16*>(weight),
                               static_cast<const __nv_bfloat16*>(bias),
                               static_cast<__nv_bfloat16*>(out), N, I, O, epi, plan, stream);
  }
  return forward_launch_simt(feats, nbr, weight, bias, out, N, I, O, dtype, epi, plan, stream);
}
}  // namespace

int subm3d_forward_ex(const void* feats, const int32_t* nbr, const void* weight, const void* bias,
                      const void* residual, subm3d_act act, void* out, int64_t N, int32_t I,
                      int32_t O, subm3d_dtype dtype, cudaStream_t stream) {
  clear_error();
  return forward_dispatch("subm3d_forward", feats, nbr, weight, bias, residual, act, out, N, I, O,
                          dtype, TilePlan{nullptr, nullptr}, stream);
}

namespace {
// The gather form subm3d_forward_grouped uses on a plan, noted per (device, buffer) when
// the plan is built: plans of windows below 4096 voxels keep most offsets per tile and
// run faster with per-thread row loads, sparser ones with staged whole-row copies. Only a
// performance choice: a buffer not noted here (a copied plan, say) gets the staged form.
constexpr int64_t kDenseWindowBelow = 4096;
std::mutex g_plan_mu;
std::map<std::pair<int, const void*>, bool> g_plan_dense;

void note_plan(const void* plan, bool dense) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(g_plan_mu);
  if (g_plan_dense.size() > 4096) g_plan_dense.clear();   // bounded: notes are only hints
  g_plan_dense[{dev, plan}] = dense;
}
bool plan_is_dense(const void* plan) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(g_plan_mu);
  const auto it = g_plan_dense.find({dev, plan});
  return it != g_plan_dense.end() && it->second;
}
}  // namespace

size_t subm3d_plan_bytes(int64_t N) {
  if (N < 0 || N > 0x7FFFFFFFll) return 0;
  return plan_layout(N).total;
}

size_t subm3d_kmap_grouped_workspace_bytes(int64_t N) { return kmap_grouped_workspace_bytes(N); }

int subm3d_build_kmap_grouped(const int32_t* coords, int64_t N, int32_t res, int64_t window,
                              void* plan, size_t plan_bytes, void* workspace, size_t ws_bytes,
                              unsigned flags, cudaStream_t stream) {
  clear_error();
  if (flags & ~static_cast<unsigned>(SUBM3D_KMAP_ASYNC)) {
    set_error("subm3d_build_kmap_grouped: unknown flags 0x%x", flags);
    return SUBM3D_ERR_ARG;
  }
  const int rc = kmap_build_grouped(coords, N, res, window, plan, plan_bytes, workspace, ws_bytes,
                                   !(flags & SUBM3D_KMAP_ASYNC), stream);
  if (rc == SUBM3D_OK && plan)
    note_plan(plan, (window ? window : SUBM3D_GROUP_WINDOW) < kDenseWindowBelow);
  return rc;
}

int subm3d_build_kmap_async(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                            void* workspace, size_t ws_bytes, cudaStream_t stream) {
  clear_error();
  return kmap_build_async(coords, N, res, nbr, workspace, ws_bytes, stream);
}

int subm3d_forward_grouped(const void* feats, const void* plan, const void* weight,
                           const void* bias, const void* residual, subm3d_act act, void* out,
                           int64_t N, int32_t I, int32_t O, subm3d_dtype dtype,
                           cudaStream_t stream) {
  clear_error();
  if (N > 0 && (!plan || (reinterpret_cast<uintptr_t>(plan) & 255))) {
    set_error("subm3d_forward_grouped: plan=%p must be a 256-byte aligned tile plan", plan);
    return SUBM3D_ERR_ARG;
  }
  if (N < 0 || N > 0x7FFFFFFFll) {
    set_error("subm3d_forward_grouped: N=%lld outside [0, 2^31)", (long long)N);
    return SUBM3D_ERR_ARG;
  }
  const PlanLayout PL = plan_layout(N);
  const char* pl = static_cast<const char*>(plan);
  const TilePlan tp{N > 0 ? reinterpret_cast<const int32_t*>(pl + PL.perm) : nullptr,
                    N > 0 ? reinterpret_cast<const uint32_t*>(pl + PL.tmask) : nullptr,
                    N > 0 && plan_is_dense(plan)};
  return forward_dispatch("subm3d_forward_grouped", feats,
                          N > 0 ? reinterpret_cast<const int32_t*>(pl + PL.nbr) : nullptr, weight,
                          bias, residual, act, out, N, I, O, dtype, tp, stream);
}


int subm3d_forward(const void* feats, const int32_t* nbr, const void* weight, const void* bias,
                   void* out, int64_t N, int32_t I, int32_t O, subm3d_dtype dtype,
                   cudaStream_t stream) {
  return subm3d_forward_ex(feats, nbr, weight, bias, nullptr, SUBM3D_ACT_NONE, out, N, I, O,
                           dtype, stream);
}

size_t subm3d_downsample_workspace_bytes(int64_t N) { return downsample_workspace_bytes(N); }

int subm3d_downsample(const int32_t* coords, int64_t N, int32_t res, const void* feats, int32_t C,
                      subm3d_dtype dtype, subm3d_pool mode, int32_t* coarse_coords,
                      void* coarse_feats, int32_t* parent, uint8_t* child_mask, int64_t* M_out,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  clear_error();
  return downsample_build(coords, N, res, nullptr, feats, C, dtype, static_cast<int>(mode),
                          coarse_coords, coarse_feats, parent, child_mask, M_out, workspace,
                          ws_bytes, stream);
}

int subm3d_downsample_sorted(const int32_t* coords, int64_t N, int32_t res, const int32_t* order,
                             const void* feats, int32_t C, subm3d_dtype dtype, subm3d_pool mode,
                             int32_t* coarse_coords, void* coarse_feats, int32_t* parent,
                             uint8_t* child_mask, int64_t* M_out, void* workspace,
                             size_t ws_bytes, cudaStream_t stream) {
  clear_error();
  if (!order && N > 0) {
    set_error("subm3d_downsample_sorted: order is NULL");
    return SUBM3D_ERR_ARG;
  }
  return downsample_build(coords, N, res, order, feats, C, dtype, static_cast<int>(mode),
                          coarse_coords, coarse_feats, parent, child_mask, M_out, workspace,
                          ws_bytes, stream);
}

int subm3d_downsample_async(const int32_t* coords, int64_t N, int32_t res, const int32_t* order,
                            const void* feats, int32_t C, subm3d_dtype dtype, subm3d_pool mode,
                            int32_t* coarse_coords, void* coarse_feats, int32_t* parent,
                            uint8_t* child_mask, int64_t* M, void* workspace, size_t ws_bytes,
                            cudaStream_t stream) {
  clear_error();
  if (!M) {
    set_error("subm3d_downsample_async: M (device) is NULL");
    return SUBM3D_ERR_ARG;
  }
  return downsample_build(coords, N, res, order, feats, C, dtype, static_cast<int>(mode),
                          coarse_coords, coarse_feats, parent, child_mask, nullptr, workspace,
                          ws_bytes, stream, M);
}

int subm3d_upsample(const void* coarse_feats, int64_t M, int32_t C, const int32_t* parent,
                    int64_t N, subm3d_dtype dtype, void* fine_feats, cudaStream_t stream) {
  clear_error();
  return upsample_launch(coarse_feats, M, C, parent, N, dtype, fine_feats, stream);
}

int subm3d_spatial2channel(const void* feats, const int32_t* coords, const int32_t* parent,
                           const uint8_t* child_mask, int64_t N, int64_t M, int32_t C,
                           subm3d_dtype dtype, void* out, cudaStream_t stream) {
  clear_error();
  return spatial2channel_launch(feats, coords, parent, child_mask, N, M, C, dtype, out, stream);
}

int subm3d_channel2spatial(const void* coarse_feats, const int32_t* coords, const int32_t* parent,
                           int64_t N, int64_t M, int32_t C, subm3d_dtype dtype, void* fine_feats,
                           cudaStream_t stream) {
  clear_error();
  return channel2spatial_launch(coarse_feats, coords, parent, N, M, C, dtype, fine_feats, stream);
}

int subm3d_forward_status(cudaStream_t stream) {
  clear_error();
  SUBM3D_CUDA_TRY(cudaStreamSynchronize(stream));
  int* word = forward_error_word();
  if (!word) return SUBM3D_ERR_CUDA;
  int host = 0;
  const int zero = 0;
  SUBM3D_CUDA_TRY(cudaMemcpy(&host, word, sizeof(int), cudaMemcpyDeviceToHost));
  SUBM3D_CUDA_TRY(cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice));
  if (host == 0) return SUBM3D_OK;
  set_error("subm3d_forward_status: device reported%s%s%s%s%s%s%s%s%s",
            (host & kDevErrBadOrder) ? " [downsample] an order that is not the Morton order" : "",
            (host & kDevErrBadNbr) ? " an nbr entry outside [-1, N)" : "",
            (host & kDevErrTimeout) ? " a pipeline wait that ran out (kernel stopped early)" : "",
            (host & kDevErrBadParent) ? " a parent entry outside [0, M)" : "",
            (host & kDevErrBadPlan) ? " a tile-plan row naming no input row" : "",
            (host & kDevErrKmapCoord) ? " [kernel map] a coordinate outside the grid" : "",
            (host & kDevErrKmapDup) ? " [kernel map] a duplicate coordinate" : "",
            (host & kDevErrKmapFull) ? " [kernel map] a full hash table" : "",
            (host & kDevErrKmapInternal) ? " [kernel map] an internal index error" : "");
  if (host & (kDevErrKmapCoord | kDevErrKmapDup | kDevErrKmapFull | kDevErrKmapInternal)) {
    if (host & kDevErrKmapCoord) return SUBM3D_ERR_COORD_RANGE;
    if (host & kDevErrKmapDup) return SUBM3D_ERR_DUPLICATE;
    if (host & kDevErrKmapFull) return SUBM3D_ERR_HASH_FULL;
  }
  if (host & kDevErrBadOrder) return SUBM3D_ERR_ARG;
  return SUBM3D_ERR_DEVICE;
}

void subm3d_kmap_stage_timing(int enable) { kmap_stage_timing(enable != 0); }

int subm3d_kmap_stage_times(float* ms, const char** names, int max) {
  clear_error();
  if (!ms || !names || max < 0) {
    set_error("subm3d_kmap_stage_times: ms=%p names=%p max=%d", (void*)ms, (void*)names, max);
    return SUBM3D_ERR_ARG;
  }
  return kmap_stage_times(ms, names, max);
}

const char* subm3d_last_error(void) { return g_msg; }

int64_t subm3d_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
