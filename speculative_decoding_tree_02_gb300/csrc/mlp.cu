// blockpilot_mlp: BlockPilot's block-size predictor (BlockPilot page §3: the
// last-prefill next-token distribution feeds a two-layer MLP that picks the
// block size once per request; §7 raw probabilities as input; §4 hidden 2048;
// §2 candidates B-3 .. B+3).
//
// Layer 1 is a bandwidth-bound GEMV with 8 right-hand sides (the requests):
// every W1 element is read once and used for 8 FMAs.  Grid (column block of
// 256 hidden units, V-slice, request group of 8).  The softmax is fused: the
// CTA first turns its slice of each request's logits into probabilities
// x = 2^((l - lse) log2 e) in shared memory.  Warps take W1 rows round-robin,
// lanes own 8 hidden units (one 16-byte load per row), and the 8 warps'
// partial sums are reduced through shared memory in warp order.  Layer 2,
// ReLU and the argmax run in one small CTA per request, summing the V-slices
// in slice order (deterministic).
#include <algorithm>

#include "tv_common.cuh"

namespace tv {

constexpr int kMThreads = 256;
constexpr int kMCols = 256;        // hidden units per CTA (8 per lane, 32 lanes)
constexpr int kMReq = 8;           // requests per CTA
constexpr int kMSub = 256;         // rows of x staged at a time

__global__ void __launch_bounds__(kMThreads) mlp_l1_kernel(
    const uint16_t* __restrict__ logits, int64_t ld, const float* __restrict__ row_lse,
    const uint16_t* __restrict__ W1, int B, int V, int H, int rows_per_slice,
    float* __restrict__ part) {
  __shared__ __align__(16) float s_x[kMSub][kMReq];
  __shared__ float s_red[kMThreads / 32][kMCols];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cb = blockIdx.x, slice = blockIdx.y, rg = blockIdx.z;
  const int v0 = slice * rows_per_slice;
  const int v1 = min(V, v0 + rows_per_slice);
  const int nb = min(kMReq, B - rg * kMReq);
  const int col0 = cb * kMCols + lane * 8;

  float acc[kMReq][8];
#pragma unroll
  for (int b = 0; b < kMReq; ++b)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[b][c] = 0.f;

  for (int s0 = v0; s0 < v1; s0 += kMSub) {
    __syncthreads();
    {
      const int v = s0 + tid;
#pragma unroll
      for (int b = 0; b < kMReq; ++b) {
        float x = 0.f;
        if (b < nb && v < v1) {
          const int rq = rg * kMReq + b;
          const float l = bf16_at(logits + static_cast<int64_t>(rq) * ld + v);
          x = ex2(fmaf(l, kLog2e, -row_lse[rq] * kLog2e));
        }
        s_x[tid][b] = x;
      }
    }
    __syncthreads();
    const int n = min(kMSub, v1 - s0);
    for (int j = warp; j < n; j += kMThreads / 32) {
      const uint4 w = ldg_stream(W1 + static_cast<int64_t>(s0 + j) * H + col0);
      const float wf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                           bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
      const float4 xa = *reinterpret_cast<const float4*>(&s_x[j][0]);
      const float4 xb = *reinterpret_cast<const float4*>(&s_x[j][4]);
      const float xs[kMReq] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int b = 0; b < kMReq; ++b)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[b][c] = fmaf(xs[b], wf[c], acc[b][c]);
    }
  }
  // reduce the 8 warps' partials, one request at a time, in warp order
  for (int b = 0; b < nb; ++b) {
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 8; ++c) s_red[warp][lane * 8 + c] = acc[b][c];
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kMThreads / 32; ++w) t += s_red[w][tid];
    const int rq = rg * kMReq + b;
    part[(static_cast<int64_t>(slice) * B + rq) * H + cb * kMCols + tid] = t;
  }
}

__global__ void __launch_bounds__(256) mlp_l2_kernel(
    const float* __restrict__ part, int n_slice, int B, int H, int C,
    const float* __restrict__ b1, const uint16_t* __restrict__ W2, const float* __restrict__ b2,
    int block, float* __restrict__ z, int32_t* __restrict__ choice, int32_t* __restrict__ bsize) {
  __shared__ float s_z[256 / 32][32];
  const int rq = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float zc[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) zc[c] = 0.f;
  for (int h = tid; h < H; h += blockDim.x) {
    float a = b1 ? b1[h] : 0.f;
    for (int s = 0; s < n_slice; ++s) a += part[(static_cast<int64_t>(s) * B + rq) * H + h];
    a = fmaxf(a, 0.f);
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (c < C) zc[c] = fmaf(a, bf16_at(W2 + static_cast<int64_t>(h) * C + c), zc[c]);
  }
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float v = warp_sum(zc[c]);
    if (lane == 0) s_z[warp][c] = v;
  }
  __syncthreads();
  if (tid == 0) {
    int best = 0;
    float bv = -INFINITY;
    for (int c = 0; c < C; ++c) {
      float v = b2 ? b2[c] : 0.f;
      for (int w = 0; w < 256 / 32; ++w) v += s_z[w][c];
      z[static_cast<int64_t>(rq) * C + c] = v;
      if (v > bv) { bv = v; best = c; }
    }
    choice[rq] = best;
    bsize[rq] = block - (C - 1) / 2 + best;
  }
}

int mlp_slices(int V, int H, int B) {
  int dev = 0, n_sm = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const int ctas_per_slice = (H / kMCols) * ((B + kMReq - 1) / kMReq);
  int s = (4 * n_sm + ctas_per_slice - 1) / ctas_per_slice;
  s = std::max(1, std::min(s, (V + kMSub - 1) / kMSub));
  return s;
}

}  // namespace tv

TV_API size_t blockpilot_mlp_workspace_size(int B, int V, int H) {
  if (B <= 0 || V <= 0 || H <= 0) return 0;
  return static_cast<size_t>(tv::mlp_slices(V, H, B)) * B * H * sizeof(float);
}

TV_API int blockpilot_mlp(const void* last_logits, int64_t ld, const float* row_lse,
                          const void* W1, const float* b1, const void* W2, const float* b2, int B,
                          int V, int H, int C, int block, float* z, int32_t* choice,
                          int32_t* bsize, void* ws, size_t ws_bytes, tv_stream_t stream) {
  if (B < 0 || V <= 0 || H <= 0 || C <= 0 || ld < V) return TV_EINVAL;
  if (H % tv::kMCols != 0 || C > 32 || B > 16) return TV_EUNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!last_logits || !row_lse || !W1 || !W2 || !z || !choice || !bsize) return TV_EINVAL;
  if (!tv::aligned(W1, 16)) return TV_EINVAL;
  const size_t need = blockpilot_mlp_workspace_size(B, V, H);
  if (!ws || ws_bytes < need || !tv::aligned(ws, 16)) return TV_EWORKSPACE;
  const int n_slice = tv::mlp_slices(V, H, B);
  const int rows_per_slice = (V + n_slice - 1) / n_slice;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  dim3 g1(H / tv::kMCols, n_slice, (B + tv::kMReq - 1) / tv::kMReq);
  tv::mlp_l1_kernel<<<g1, tv::kMThreads, 0, st>>>(
      static_cast<const uint16_t*>(last_logits), ld, row_lse, static_cast<const uint16_t*>(W1), B,
      V, H, rows_per_slice, static_cast<float*>(ws));
  tv::mlp_l2_kernel<<<B, 256, 0, st>>>(static_cast<const float*>(ws), n_slice, B, H, C, b1,
                                       static_cast<const uint16_t*>(W2), b2, block, z, choice,
                                       bsize);
  return tv::launch_status();
}
