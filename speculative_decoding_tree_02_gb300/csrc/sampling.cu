// accept_rejection_sampling: lossless temperature-1 verification of a draft
// tree (SpecOPD page §03: acceptance under exact rejection sampling is the
// draft/target overlap; D-cut page §4, SpecOPD page §04: T = 1 results).
// Scheme (the pages give none): children in index order are accepted with
// probability min(1, p'(x)/q(x)); after each rejection p' becomes the
// normalised residual max(0, p' - q); with no child accepted the bonus token
// is drawn from p' by inverse CDF.  Uniforms are inputs.
//
// One CTA of 1024 threads per request walks the tree; every distribution
// operation is a pass over the vocabulary: log-sum-exp of the target and
// draft rows of the current node (one online pass), a residual pass per
// rejection (written to the request's fp32 workspace row), and a prefix-sum
// search for the bonus token.  Exponentials and per-thread sums in fp32,
// cross-warp sums in fp64.
#include <cuda_bf16.h>

#include <algorithm>

#include "tv_common.cuh"

namespace tv {

constexpr int kRsThreads = 1024;

template <typename T>
__device__ __forceinline__ float rs_val(const T* row, int v) {
  if constexpr (sizeof(T) == 2) return bf16_at(reinterpret_cast<const uint16_t*>(row) + v);
  else return reinterpret_cast<const float*>(row)[v];
}

// Sum over the 1024 threads: fp32 within a warp, fp64 across the 32 warps
// (fp64 is scarce on this part; a warp's 32 terms lose nothing that matters).
__device__ __forceinline__ double rs_sum(float v, double* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll 4
  for (int w = 0; w < kRsThreads / 32; ++w) t += s_red[w];
  return t;
}

__device__ __forceinline__ float rs_max(float v, float* s_m) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) s_m[warp] = v;
  __syncthreads();
  float t = s_m[0];
  for (int w = 1; w < kRsThreads / 32; ++w) t = fmaxf(t, s_m[w]);
  return t;
}

template <typename T>
__global__ void __launch_bounds__(kRsThreads) rejection_kernel(
    const int32_t* __restrict__ parent, const int32_t* __restrict__ tok, const T* __restrict__ pl,
    const T* __restrict__ ql, int V, int64_t ld, const int32_t* __restrict__ node_off, int max_depth,
    const float* __restrict__ u_node, const float* __restrict__ u_final, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ best_node, int32_t* __restrict__ path, int32_t* __restrict__ bonus,
    float* __restrict__ buf_all) {
  __shared__ int16_t s_first[TV_MAX_NODES], s_next[TV_MAX_NODES];
  __shared__ double s_red[32];
  __shared__ float s_m[32];
  __shared__ double s_scan[kRsThreads / 32];
  __shared__ int s_pick;
  griddep_wait();
  griddep_release();
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = node_off[r];
  const int n = min(node_off[r + 1] - n0, TV_MAX_NODES);
  float* buf = buf_all + static_cast<int64_t>(r) * V;
  for (int i = tid; i < n; i += kRsThreads) { s_first[i] = -1; s_next[i] = -1; }
  __syncthreads();
  if (tid == 0) {   // child lists in index order
    for (int i = n - 1; i >= 1; --i) {
      const int p = parent[n0 + i];
      if (p >= 0 && p < i) { s_next[i] = s_first[p]; s_first[p] = static_cast<int16_t>(i); }
    }
  }
  for (int d = tid; d <= max_depth; d += kRsThreads)
    path[static_cast<int64_t>(r) * (max_depth + 1) + d] = d == 0 ? 0 : -1;
  __syncthreads();
  int cur = 0, depth = 0;
  for (;;) {
    const T* prow = pl + static_cast<int64_t>(n0 + cur) * ld;
    const T* qrow = ql + static_cast<int64_t>(n0 + cur) * ld;
    // log-sum-exp of both rows: maxima, then sums of exp (base 2 on the SFU)
    float mp = -INFINITY, mq = -INFINITY;
    for (int v = tid; v < V; v += kRsThreads) { mp = fmaxf(mp, rs_val(prow, v)); mq = fmaxf(mq, rs_val(qrow, v)); }
    mp = rs_max(mp, s_m);
    mq = rs_max(mq, s_m);
    float sp = 0.f, sq = 0.f;
    for (int v = tid; v < V; v += kRsThreads) {
      sp += ex2((rs_val(prow, v) - mp) * kLog2e);
      sq += ex2((rs_val(qrow, v) - mq) * kLog2e);
    }
    const double Sp = rs_sum(sp, s_red), Sq = rs_sum(sq, s_red);
    // p(v) = 2^(pl(v) log2e - bp), q(v) likewise
    const float bp = static_cast<float>((mp + log(Sp)) * static_cast<double>(kLog2e));
    const float bq = static_cast<float>((mq + log(Sq)) * static_cast<double>(kLog2e));
    bool resid = false;   // p' = buf * inv_z once a child was rejected
    float inv_z = 1.f;
    int next = -1;
    for (int c = s_first[cur]; c >= 0; c = s_next[c]) {
      const int x = tok[n0 + c];
      const bool xin = x >= 0 && x < V;
      const float qx = xin ? ex2(fmaf(rs_val(qrow, x), kLog2e, -bq)) : 0.f;
      const float px = !xin ? 0.f : resid ? buf[x] * inv_z : ex2(fmaf(rs_val(prow, x), kLog2e, -bp));
      const float ratio = qx <= 0.f ? 1.f : fminf(1.f, px / qx);
      if (u_node[n0 + c] < ratio) { next = c; break; }
      // residual max(0, p' - q) into buf, and its sum
      float z = 0.f;
      for (int v = tid; v < V; v += kRsThreads) {
        const float pv = resid ? buf[v] * inv_z : ex2(fmaf(rs_val(prow, v), kLog2e, -bp));
        const float qv = ex2(fmaf(rs_val(qrow, v), kLog2e, -bq));
        const float w = fmaxf(0.f, pv - qv);
        buf[v] = w;
        z += w;
      }
      const double Z = rs_sum(z, s_red);   // (its barriers also order buf)
      if (Z > 0.0) {
        resid = true;
        inv_z = static_cast<float>(1.0 / Z);
      } else {
        resid = false;   // degenerate (rounding only): back to the target softmax
      }
    }
    if (next < 0) {
      // bonus token: smallest j with cumulative p'(<= j) > u * total, over
      // contiguous per-thread segments in token order
      const int seg = (V + kRsThreads - 1) / kRsThreads;
      const int v0 = min(V, tid * seg), v1 = min(V, v0 + seg);
      float part = 0.f;
      for (int v = v0; v < v1; ++v) part += resid ? buf[v] : ex2(fmaf(rs_val(prow, v), kLog2e, -bp));
      float inc = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) s_scan[warp] = inc;
      if (tid == 0) s_pick = V - 1;
      __syncthreads();
      double wbase = 0.0, total = 0.0;
      for (int w = 0; w < kRsThreads / 32; ++w) {
        if (w < warp) wbase += s_scan[w];
        total += s_scan[w];
      }
      const double lo = wbase + static_cast<double>(inc - part);
      const double target = static_cast<double>(u_final[r]) * total;
      if (part > 0.f && lo <= target && target < lo + part) {
        double cum = lo;
        int j = v1 - 1;
        for (int v = v0; v < v1; ++v) {
          cum += resid ? buf[v] : ex2(fmaf(rs_val(prow, v), kLog2e, -bp));
          if (cum > target) { j = v; break; }
        }
        atomicMin(&s_pick, j);
      }
      __syncthreads();
      if (tid == 0) {
        bonus[r] = s_pick;
        accept_len[r] = depth;
        best_node[r] = cur;
      }
      return;
    }
    cur = next;
    ++depth;
    if (tid == 0 && depth <= max_depth) path[static_cast<int64_t>(r) * (max_depth + 1) + depth] = cur;
    __syncthreads();
  }
}

}  // namespace tv

TV_API size_t accept_rejection_sampling_workspace_size(int B, int V) {
  if (B <= 0 || V <= 0) return 0;
  return static_cast<size_t>(B) * V * sizeof(float);
}

TV_API int accept_rejection_sampling(const int32_t* parent, const int32_t* tok, const void* p_logits,
                                     const void* q_logits, int dtype, int V, int64_t ld, const int32_t* node_off,
                                     int B, int max_nodes, int max_depth, const float* u_node,
                                     const float* u_final, int32_t* accept_len, int32_t* best_node, int32_t* path,
                                     int32_t* bonus, void* ws, size_t ws_bytes, tv_stream_t stream) {
  if (B < 0 || V <= 0 || ld < V || max_nodes < 0 || max_depth < 0) return TV_EINVAL;
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_EINVAL;
  if (max_nodes > TV_MAX_NODES) return TV_EUNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!parent || !tok || !p_logits || !q_logits || !node_off || !u_node || !u_final || !accept_len ||
      !best_node || !path || !bonus)
    return TV_EINVAL;
  if (!ws || ws_bytes < accept_rejection_sampling_workspace_size(B, V) || !tv::aligned(ws, 16)) return TV_EWORKSPACE;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  auto* buf = static_cast<float*>(ws);
  if (dtype == TV_BF16)
    return tv::launch_pdl(tv::rejection_kernel<uint16_t>, dim3(B), dim3(tv::kRsThreads), 0, st, parent, tok,
                          static_cast<const uint16_t*>(p_logits), static_cast<const uint16_t*>(q_logits), V, ld,
                          node_off, max_depth, u_node, u_final, accept_len, best_node, path, bonus, buf);
  return tv::launch_pdl(tv::rejection_kernel<float>, dim3(B), dim3(tv::kRsThreads), 0, st, parent, tok,
                        static_cast<const float*>(p_logits), static_cast<const float*>(q_logits), V, ld, node_off,
                        max_depth, u_node, u_final, accept_len, best_node, path, bonus, buf);
}
