// Forward pass on the CUDA cores: the fp32 path, and bf16 shapes outside the
// tensor-core kernel (O > 256). Output-stationary like the tensor-core kernel: a
// block owns 32 output rows x 64 output columns, walks the 27 offsets, stages the
// gathered neighbour rows and the matching weight slice in shared memory in
// 32-channel chunks, and accumulates in fp32 registers. Each output element is
// written once.
//
// out[i, o] = bias[o] + sum_k sum_c W[o, kz, ky, kx, c] * feats[nbr[i, k], c]
// (submanifold convolution, kernel 3, stride 1, no padding; weight [O, kz, ky, kx, I]
// as in the "pixal3d_mrp_mlx README" commit header).
#include "common.cuh"

namespace subm3d {
namespace {

constexpr int kRows = 32;
constexpr int kCols = 64;
constexpr int kChunk = 32;
constexpr int kThreads = 256;
constexpr int kRowsPerThread = kRows / (kThreads / kCols);   // 8

__device__ __forceinline__ float load_f(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(kThreads) fwd_simt(const T* __restrict__ feats,
                                                     const int32_t* __restrict__ nbr,
                                                     const T* __restrict__ weight,
                                                     const T* __restrict__ bias, T* __restrict__ out,
                                                     int64_t N, int I, int O, int* err) {
  __shared__ float g[kRows][kChunk + 1];
  __shared__ float w[kChunk][kCols];
  __shared__ int jrow[kRows];
  const int tid = threadIdx.x;
  const int ol = tid % kCols;
  const int r4 = tid / kCols;
  const int64_t row0 = blockIdx.x * int64_t(kRows);
  const int o = blockIdx.y * kCols + ol;
  float acc[kRowsPerThread];
#pragma unroll
  for (int m = 0; m < kRowsPerThread; ++m) acc[m] = 0.f;
  bool bad = false;
  for (int k = 0; k < 27; ++k) {
    int j = -1;
    if (tid < kRows) {
      const int64_t i = row0 + tid;
      if (i < N) {
        j = nbr[i * 27 + k];
        if (j < -1 || j >= N) {
          bad = true;
          j = -1;
        }
      }
      jrow[tid] = j;
    }
    if (!__syncthreads_or(j >= 0)) continue;
    for (int c0 = 0; c0 < I; c0 += kChunk) {
      for (int e = tid; e < kRows * kChunk; e += kThreads) {
        const int r = e / kChunk, cc = e % kChunk, c = c0 + cc;
        const int jj = jrow[r];
        g[r][cc] = (jj >= 0 && c < I) ? load_f(feats + int64_t(jj) * I + c) : 0.f;
      }
      for (int e = tid; e < kChunk * kCols; e += kThreads) {
        const int cc = e / kCols, oo = blockIdx.y * kCols + e % kCols, c = c0 + cc;
        w[cc][e % kCols] = (oo < O && c < I) ? load_f(weight + (int64_t(oo) * 27 + k) * I + c) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int cc = 0; cc < kChunk; ++cc) {
        const float wv = w[cc][ol];
#pragma unroll
        for (int m = 0; m < kRowsPerThread; ++m) acc[m] = fmaf(g[r4 + 4 * m][cc], wv, acc[m]);
      }
      __syncthreads();
    }
  }
  if (bad) atomicOr(err, kDevErrBadNbr);
  if (o >= O) return;
  const float bv = bias ? load_f(bias + o) : 0.f;
#pragma unroll
  for (int m = 0; m < kRowsPerThread; ++m) {
    const int64_t i = row0 + r4 + 4 * m;
    if (i < N) store_f(out + i * O + o, acc[m] + bv);
  }
}

}  // namespace

int forward_launch_simt(const void* feats, const int32_t* nbr, const void* weight,
                        const void* bias, void* out, int64_t N, int I, int O, subm3d_dtype dtype,
                        cudaStream_t stream) {
  const int64_t tiles = (N + kRows - 1) / kRows;
  if (tiles > 0x7FFFFFFFll) {
    set_error("subm3d_forward: N=%lld too large for the CUDA-core kernel", (long long)N);
    return SUBM3D_ERR_UNSUPPORTED;
  }
  dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>((O + kCols - 1) / kCols));
  if (dtype == SUBM3D_F32) {
    fwd_simt<float><<<grid, kThreads, 0, stream>>>(
        static_cast<const float*>(feats), nbr, static_cast<const float*>(weight),
        static_cast<const float*>(bias), static_cast<float*>(out), N, I, O, forward_error_word());
  } else {
    fwd_simt<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(feats), nbr, static_cast<const __nv_bfloat16*>(weight),
        static_cast<const __nv_bfloat16*>(bias), static_cast<__nv_bfloat16*>(out), N, I, O,
        forward_error_word());
  }
  SUBM3D_LAUNCHED("fwd_simt");
  return SUBM3D_OK;
}

}  // namespace subm3d
