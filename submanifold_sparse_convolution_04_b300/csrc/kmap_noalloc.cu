// subm3d_build_kmap_noalloc: the kernel-map build for callers that cannot allocate
// device memory, with its scratch space in a fixed array compiled into this library.
//
// Some callers cannot call cudaMalloc (or have torch allocate for them): a host
// application that owns every byte of device memory through its own pool and hands
// plugins only their input and output buffers, or a latency-critical loop in which an
// allocation (which may synchronise the device) is not acceptable. They still pass
// coords and nbr; the hash table, sort buffers and status word that
// subm3d_build_kmap keeps in the caller's workspace live here instead, in
// g_kmap_scratch, sized for at most kNoAllocMaxVoxels voxels.
//
// g_kmap_scratch is a file-scope __device__ array: every GPU that loads the library
// holds its 16 MiB until the process exits. In host code its name is only a host-side
// stand-in, so its device address is fetched with cudaGetSymbolAddress, once per
// device, with that device current, by the first call made on that device. Like
// subm3d_build_kmap, each call waits for its stream at its end (it reads the build's
// status back), so no call can be stream-captured, and two calls from one host thread
// never overlap on the GPU. All calls share the array and the build re-initialises everything it reads,
// so each call starts clean; calls made at the same time from several host threads race
// on it.
#include <mutex>

#include "common.cuh"

namespace subm3d {
namespace {

constexpr int64_t kNoAllocMaxVoxels = SUBM3D_NOALLOC_MAX_VOXELS;
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_kmap_scratch[kNoAllocScratchBytes];

PerDevice<void*> g_scratch_ptr;

// Device address of g_kmap_scratch on the current device (looked up once per device).
int scratch_on_current_device(void** out) {
  return g_scratch_ptr.get(out, [](void** v) -> int {
    void* p = nullptr;
    SUBM3D_CUDA_TRY(cudaGetSymbolAddress(&p, g_kmap_scratch));
    *v = p;
    return static_cast<int>(SUBM3D_OK);
  });
}

}  // namespace
}  // namespace subm3d

using namespace subm3d;

extern "C" int subm3d_build_kmap_noalloc(const int32_t* coords, int64_t N, int32_t res,
                                         int32_t* nbr, cudaStream_t stream) {
  clear_error();
  if (N < 0 || N > kNoAllocMaxVoxels) {
    set_error("subm3d_build_kmap_noalloc: N=%lld outside [0, %lld] (the built-in scratch holds "
              "at most %lld voxels; use subm3d_build_kmap with a workspace for more)",
              (long long)N, (long long)kNoAllocMaxVoxels, (long long)kNoAllocMaxVoxels);
    return SUBM3D_ERR_ARG;
  }
  if (N == 0) return kmap_build(coords, 0, res, nbr, nullptr, 0, nullptr, 0, stream);
  const size_t need = kmap_workspace_bytes(N, 0);
  if (need > kNoAllocScratchBytes) {
    set_error("subm3d_build_kmap_noalloc: N=%lld needs %zu scratch bytes, %zu built in",
              (long long)N, need, kNoAllocScratchBytes);
    return SUBM3D_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != SUBM3D_OK) return rc;
  return kmap_build(coords, N, res, nbr, nullptr, 0, scratch, kNoAllocScratchBytes, stream);
}
