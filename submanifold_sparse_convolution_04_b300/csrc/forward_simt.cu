// Forward pass on the CUDA cores: the fp32 path, and bf16 shapes outside the
// tensor-core kernels (O > 256). Output-stationary like the tensor-core kernels: a
// block owns 32 output rows x 64 output columns, stages its 32 x 27 block of nbr in
// shared memory once, lists the offsets at which any of its rows has a neighbour, and
// walks those offsets in 32-channel chunks: the gathered neighbour rows and the
// matching weight slice go through shared memory, and each thread accumulates 8 rows
// of one column in fp32 registers. The next step's operands are loaded into registers
// while the current step computes, so a step costs about one memory latency, not the
// three dependent ones (index, row, weight) of a plain loop. Each output element is
// written once, after the fused epilogue (+ bias [+ residual], activation).
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
constexpr int kGPerThread = kRows * kChunk / kThreads;       // 4
constexpr int kWPerThread = kChunk * kCols / kThreads;       // 8

// Read-only operands (feats, weight, bias) through the non-coherent path.
__device__ __forceinline__ float load_ro(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_ro(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }
// The residual may be the output buffer itself: plain loads.
__device__ __forceinline__ float load_rw(const float* p) { return *p; }
__device__ __forceinline__ float load_rw(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(kThreads) fwd_simt(const T* __restrict__ feats,
                                                     const int32_t* __restrict__ nbr,
                                                     const T* __restrict__ weight,
                                                     const T* __restrict__ bias, const T* residual,
                                                     int act, T* out, int64_t N, int I, int O,
                                                     int* err, const int32_t* __restrict__ perm) {
  __shared__ float g[kRows][kChunk + 1];     // gathered rows of one step
  __shared__ float w[kChunk][kCols + 1];     // weight slice of one step
  __shared__ int32_t jt[kRows * 27];         // this block's rows of nbr
  __shared__ int ks[27];                     // offsets with at least one neighbour
  __shared__ int nks;
  const int tid = threadIdx.x;
  const int ol = tid % kCols;
  const int r4 = tid / kCols;
  const int64_t row0 = blockIdx.x * int64_t(kRows);
  const int o0 = blockIdx.y * kCols;
  const int o = o0 + ol;

  bool bad = false;
  for (int e = tid; e < kRows * 27; e += kThreads) {
    int j = -1;
    if (row0 + e / 27 < N) {
      j = nbr[row0 * 27 + e];
      if (j < -1 || j >= N) {
        bad = true;
        j = -1;
      }
    }
    jt[e] = j;
  }
  __syncthreads();
  if (tid < 32) {
    bool any = false;
    if (tid < 27)
      for (int r = 0; r < kRows; ++r) any |= jt[r * 27 + tid] >= 0;
    const unsigned m = __ballot_sync(0xffffffffu, any);
    if (any) ks[__popc(m & ((1u << tid) - 1u))] = tid;
    if (tid == 0) nks = __popc(m);
  }
  __syncthreads();

  const int nch = (I + kChunk - 1) / kChunk;
  const int nsteps = nks * nch;
  float gr[kGPerThread], wr[kWPerThread];
  auto load_step = [&](int s) {
    const int k = ks[s / nch];
    const int c0 = (s % nch) * kChunk;
#pragma unroll
    for (int q = 0; q < kGPerThread; ++q) {
      const int e = tid + q * kThreads;
      const int r = e / kChunk, c = c0 + e % kChunk;
      const int jj = jt[r * 27 + k];
      gr[q] = (jj >= 0 && c < I) ? load_ro(feats + int64_t(jj) * I + c) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kWPerThread; ++q) {
      const int e = tid + q * kThreads;
      const int oo = o0 + e / kChunk, c = c0 + e % kChunk;
      wr[q] = (oo < O && c < I) ? load_ro(weight + (int64_t(oo) * 27 + k) * I + c) : 0.f;
    }
  };

  float acc[kRowsPerThread];
#pragma unroll
  for (int m = 0; m < kRowsPerThread; ++m) acc[m] = 0.f;
  if (nsteps > 0) load_step(0);
  for (int s = 0; s < nsteps; ++s) {
#pragma unroll
    for (int q = 0; q < kGPerThread; ++q) {
      const int e = tid + q * kThreads;
      g[e / kChunk][e % kChunk] = gr[q];
    }
#pragma unroll
    for (int q = 0; q < kWPerThread; ++q) {
      const int e = tid + q * kThreads;
      w[e % kChunk][e / kChunk] = wr[q];
    }
    __syncthreads();
    if (s + 1 < nsteps) load_step(s + 1);   // in flight during the FMAs below
#pragma unroll 8
    for (int cc = 0; cc < kChunk; ++cc) {
      const float wv = w[cc][ol];
#pragma unroll
      for (int m = 0; m < kRowsPerThread; ++m) acc[m] = fmaf(g[r4 + 4 * m][cc], wv, acc[m]);
    }
    __syncthreads();
  }
  if (bad) atomicOr(err, kDevErrBadNbr);
  if (o >= O) return;
  const float bv = bias ? load_ro(bias + o) : 0.f;
#pragma unroll
  for (int m = 0; m < kRowsPerThread; ++m) {
    int64_t i = row0 + r4 + 4 * m;   // row of the tile order; with a plan, perm[i] is the output row
    if (perm && i < N) {
      i = __ldg(perm + i);
      if (i < 0 || i >= N) {
        if (ol == 0) atomicOr(err, kDevErrBadPlan);
        continue;
      }
    }
    if (i < N) {
      float y = acc[m] + bv;
      if (residual) y += load_rw(residual + i * O + o);
      store_f(out + i * O + o, apply_act(y, act));
    }
  }
}

}  // namespace

int forward_launch_simt(const void* feats, const int32_t* nbr, const void* weight,
                        const void* bias, void* out, int64_t N, int I, int O, subm3d_dtype dtype,
                        Epilogue epi, TilePlan plan, cudaStream_t stream) {
  const int64_t tiles = (N + kRows - 1) / kRows;
  if (tiles > 0x7FFFFFFFll) {
    set_error("subm3d_forward: N=%lld too large for the CUDA-core kernel", (long long)N);
    return SUBM3D_ERR_UNSUPPORTED;
  }
  int* err = forward_error_word();
  if (!err) return SUBM3D_ERR_CUDA;
  dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>((O + kCols - 1) / kCols));
  if (dtype == SUBM3D_F32) {
    fwd_simt<float><<<grid, kThreads, 0, stream>>>(
        static_cast<const float*>(feats), nbr, static_cast<const float*>(weight),
        static_cast<const float*>(bias), static_cast<const float*>(epi.residual), epi.act,
        static_cast<float*>(out), N, I, O, err, plan.perm);
  } else {
    fwd_simt<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(feats), nbr, static_cast<const __nv_bfloat16*>(weight),
        static_cast<const __nv_bfloat16*>(bias), static_cast<const __nv_bfloat16*>(epi.residual),
        epi.act, static_cast<__nv_bfloat16*>(out), N, I, O, err, plan.perm);
  }
  SUBM3D_LAUNCHED("fwd_simt");
  return SUBM3D_OK;
}

}  // namespace subm3d
