// accept_rejection_sampling: lossless temperature-1 verification of a draft
// tree (SpecOPD page §03: acceptance under exact rejection sampling is the
// draft/target overlap; D-cut page §4, SpecOPD page §04: T = 1 results).
// Scheme (the pages give none): children in index order are accepted with
// probability min(1, p'(x)/q(x)); after each rejection p' becomes the
// normalised residual max(0, p' - q); with no child accepted the bonus token
// is drawn from p' by inverse CDF.  Uniforms are inputs.
//
// A cluster of 8 CTAs per request walks the tree; every distribution
// operation is a pass over the vocabulary split into eighths: log-sum-exp of
// the target and draft rows of the current node (one online pass), a
// residual pass per rejection (written to the request's fp32 workspace row),
// and a prefix-sum search for the bonus token, with the CTAs' partials
// exchanged through distributed shared memory.  All arithmetic in fp32.
#include <cuda_bf16.h>

#include <algorithm>

#include "tv_common.cuh"

namespace tv {

constexpr int kRsCluster = 8;     // CTAs per request, each on an eighth of the vocabulary
constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;

template <typename T>
__device__ __forceinline__ float rs_val(const T* row, int v) {
  if constexpr (sizeof(T) == 2) return bf16_at(reinterpret_cast<const uint16_t*>(row) + v);
  else return reinterpret_cast<const float*>(row)[v];
}

__device__ __forceinline__ uint32_t rs_smem(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void rs_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the float at the same shared-memory offset in CTA `rank` of this cluster
__device__ __forceinline__ float rs_remote(const float* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(rs_smem(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// running (max, sum of exp(x - max)) of one value stream
__device__ __forceinline__ void rs_online(float x, float& m, float& s) {
  if (x > m) {
    s = s * ex2((m - x) * kLog2e) + 1.f;   // an empty sum (m = -inf) stays 0
    m = x;
  } else if (x != -INFINITY) {
    s += ex2((x - m) * kLog2e);
  }
}

// Per-CTA scratch of the walk.
struct RsShared {
  int16_t first[TV_MAX_NODES], next[TV_MAX_NODES];   // child lists in index order
  float xch[2][4];                                    // cluster exchange slots (by parity)
  float all[kRsCluster][4];                           // the cluster's values of the last exchange
  float wred[kRsWarps][4];
  float wmax[kRsWarps][2];
  float res[4];                                       // thread 0's combined results of a step
  int own;
  int pick;
};

// Exchange four floats with the other CTAs of the cluster: afterwards
// sh.all[c][*] holds CTA c's values in every CTA.  Exchange e uses slot e & 1;
// a CTA rewrites a slot only after the barrier of the following exchange,
// which every reader reaches after its reads.
__device__ __forceinline__ void rs_exchange(RsShared& sh, int e, float a, float b, float c, float d) {
  if (threadIdx.x == 0) {
    sh.xch[e & 1][0] = a; sh.xch[e & 1][1] = b; sh.xch[e & 1][2] = c; sh.xch[e & 1][3] = d;
  }
  rs_cluster_sync();
  if (threadIdx.x < kRsCluster * 4) {
    const int cta = threadIdx.x >> 2, f = threadIdx.x & 3;
    sh.all[cta][f] = rs_remote(&sh.xch[e & 1][f], cta);
  }
  __syncthreads();
}

// CTA sum (warp sums, then thread 0 over the warps in order); valid in
// thread 0 only.  All cross-thread arithmetic is fp32: fp64 is scarce on this
// part and a handful of partial sums loses nothing that matters.
__device__ __forceinline__ float rs_cta_sum0(RsShared& sh, float v) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) sh.wred[threadIdx.x >> 5][0] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kRsWarps; ++w) t += sh.wred[w][0];
  return t;
}

// 8 consecutive bf16 logits (16-byte aligned)
__device__ __forceinline__ void rs_online8(uint4 x, float& m, float& s) {
  const __nv_bfloat162 h = __hmax2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&x.x),
                                           *reinterpret_cast<const __nv_bfloat162*>(&x.y)),
                                   __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&x.z),
                                           *reinterpret_cast<const __nv_bfloat162*>(&x.w)));
  const float m8 = fmaxf(__low2float(h), __high2float(h));
  if (m8 > m) {
    s *= ex2((m - m8) * kLog2e);
    m = m8;
  }
  if (m != -INFINITY) {
    const float bm = m * kLog2e;
    s += ex2(fmaf(bf16_lo(x.x), kLog2e, -bm)) + ex2(fmaf(bf16_hi(x.x), kLog2e, -bm)) +
         ex2(fmaf(bf16_lo(x.y), kLog2e, -bm)) + ex2(fmaf(bf16_hi(x.y), kLog2e, -bm)) +
         ex2(fmaf(bf16_lo(x.z), kLog2e, -bm)) + ex2(fmaf(bf16_hi(x.z), kLog2e, -bm)) +
         ex2(fmaf(bf16_lo(x.w), kLog2e, -bm)) + ex2(fmaf(bf16_hi(x.w), kLog2e, -bm));
  }
}

// A cluster of 8 CTAs per request walks its tree; every CTA takes the same
// decisions (the same exchanged partials, combined in CTA order), and each
// vocabulary pass is split by slices: CTA c owns [c S, (c + 1) S).
//   node      one online pass over the slice for (max, sum of exp) of the
//             target and draft rows; exchange; lse of both rows
//   child     accept test from the two logits of its token (and the
//             residual row in the workspace); on rejection a residual pass
//             writes max(0, p' - q) of the slice and its sum; exchange
//   bonus     slice totals of p'; exchange; the CTA whose slice holds the
//             inverse-CDF target finds the token inside it
template <typename T>
__global__ void __cluster_dims__(kRsCluster, 1, 1) __launch_bounds__(kRsThreads, 4) rejection_kernel(
    const int32_t* __restrict__ parent, const int32_t* __restrict__ tok, const T* __restrict__ pl,
    const T* __restrict__ ql, int V, int64_t ld, const int32_t* __restrict__ node_off, int max_depth,
    const float* __restrict__ u_node, const float* __restrict__ u_final, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ best_node, int32_t* __restrict__ path, int32_t* __restrict__ bonus,
    float* __restrict__ buf_all, bool vec) {
  __shared__ RsShared sh;
  griddep_wait();
  griddep_release();
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int r = blockIdx.x / kRsCluster, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = node_off[r];
  const int n = min(node_off[r + 1] - n0, TV_MAX_NODES);
  const int S = ((V + kRsCluster - 1) / kRsCluster + 7) / 8 * 8;   // slice starts stay 16-byte aligned
  const int v0 = min(V, static_cast<int>(rank) * S), v1 = min(V, v0 + S);
  float* buf = buf_all + static_cast<int64_t>(r) * V;
  for (int i = tid; i < n; i += kRsThreads) { sh.first[i] = -1; sh.next[i] = -1; }
  __syncthreads();
  if (tid == 0) {
    for (int i = n - 1; i >= 1; --i) {
      const int p = parent[n0 + i];
      if (p >= 0 && p < i) { sh.next[i] = sh.first[p]; sh.first[p] = static_cast<int16_t>(i); }
    }
  }
  if (rank == 0)
    for (int d = tid; d <= max_depth; d += kRsThreads)
      path[static_cast<int64_t>(r) * (max_depth + 1) + d] = d == 0 ? 0 : -1;
  __syncthreads();
  int cur = 0, depth = 0, e = 0;
  for (;;) {
    const T* prow = pl + static_cast<int64_t>(n0 + cur) * ld;
    const T* qrow = ql + static_cast<int64_t>(n0 + cur) * ld;
    // log-sum-exp of both rows over the slice, then across the cluster
    float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
    int v = v0 + tid;
    if constexpr (sizeof(T) == 2) {
      if (vec) {   // 16-byte vectors over the slice's whole eighths, scalar tail
        const int nv = (v1 - v0) / 8;
        const uint4* vp = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(prow) + v0);
        const uint4* vq = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(qrow) + v0);
        for (int i = tid; i < nv; i += kRsThreads) {
          const uint4 x = __ldg(vp + i), y = __ldg(vq + i);
          rs_online8(x, mp, sp);
          rs_online8(y, mq, sq);
        }
        v = v0 + nv * 8 + tid;
      }
    }
    for (; v + 3 * kRsThreads < v1; v += 4 * kRsThreads) {
      float xp[4], xq[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) { xp[u] = rs_val(prow, v + u * kRsThreads); xq[u] = rs_val(qrow, v + u * kRsThreads); }
#pragma unroll
      for (int u = 0; u < 4; ++u) { rs_online(xp[u], mp, sp); rs_online(xq[u], mq, sq); }
    }
    for (; v < v1; v += kRsThreads) { rs_online(rs_val(prow, v), mp, sp); rs_online(rs_val(qrow, v), mq, sq); }
    {
      const float Mp = warp_max(mp), Mq = warp_max(mq);
      const float tp = warp_sum(mp == -INFINITY ? 0.f : sp * ex2((mp - Mp) * kLog2e));
      const float tq = warp_sum(mq == -INFINITY ? 0.f : sq * ex2((mq - Mq) * kLog2e));
      if (lane == 0) { sh.wmax[warp][0] = Mp; sh.wmax[warp][1] = Mq; sh.wred[warp][0] = tp; sh.wred[warp][1] = tq; }
    }
    __syncthreads();
    float cmp = -INFINITY, csp = 0.f, cmq = -INFINITY, csq = 0.f;
    if (tid == 0) {
      for (int w = 0; w < kRsWarps; ++w) { cmp = fmaxf(cmp, sh.wmax[w][0]); cmq = fmaxf(cmq, sh.wmax[w][1]); }
      for (int w = 0; w < kRsWarps; ++w) {
        if (sh.wmax[w][0] != -INFINITY) csp += sh.wred[w][0] * ex2((sh.wmax[w][0] - cmp) * kLog2e);
        if (sh.wmax[w][1] != -INFINITY) csq += sh.wred[w][1] * ex2((sh.wmax[w][1] - cmq) * kLog2e);
      }
    }
    rs_exchange(sh, e++, cmp, csp, cmq, csq);
    if (tid == 0) {   // p(v) = 2^(pl(v) log2e - bp), q(v) likewise
      float Mp = -INFINITY, Mq = -INFINITY;
      for (int c = 0; c < kRsCluster; ++c) { Mp = fmaxf(Mp, sh.all[c][0]); Mq = fmaxf(Mq, sh.all[c][2]); }
      float Sp = 0.f, Sq = 0.f;
      for (int c = 0; c < kRsCluster; ++c) {
        if (sh.all[c][0] != -INFINITY) Sp += sh.all[c][1] * ex2((sh.all[c][0] - Mp) * kLog2e);
        if (sh.all[c][2] != -INFINITY) Sq += sh.all[c][3] * ex2((sh.all[c][2] - Mq) * kLog2e);
      }
      sh.res[0] = Mp * kLog2e + log2f(Sp);
      sh.res[1] = Mq * kLog2e + log2f(Sq);
    }
    __syncthreads();
    const float bp = sh.res[0], bq = sh.res[1];
    bool resid = false;   // p' = buf * inv_z once a child was rejected
    float inv_z = 1.f;
    int next = -1;
    for (int c = sh.first[cur]; c >= 0; c = sh.next[c]) {
      const int x = tok[n0 + c];
      const bool xin = x >= 0 && x < V;
      const float qx = xin ? ex2(fmaf(rs_val(qrow, x), kLog2e, -bq)) : 0.f;
      const float px = !xin ? 0.f : resid ? buf[x] * inv_z : ex2(fmaf(rs_val(prow, x), kLog2e, -bp));
      const float ratio = qx <= 0.f ? 1.f : fminf(1.f, px / qx);
      if (u_node[n0 + c] < ratio) { next = c; break; }
      // residual max(0, p' - q) of the slice into buf, and its sum
      float z = 0.f;
      int w0 = v0 + tid;
      if constexpr (sizeof(T) == 2) {
        if (vec) {
          const int nv = (v1 - v0) / 8;
          const uint4* vp = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(prow) + v0);
          const uint4* vq = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(qrow) + v0);
          float4* bo = reinterpret_cast<float4*>(buf + v0);
          for (int i = tid; i < nv; i += kRsThreads) {
            const uint4 y = __ldg(vq + i);
            float pv[8];
            if (resid) {
              const float4 a = bo[2 * i], b = bo[2 * i + 1];
              pv[0] = a.x * inv_z; pv[1] = a.y * inv_z; pv[2] = a.z * inv_z; pv[3] = a.w * inv_z;
              pv[4] = b.x * inv_z; pv[5] = b.y * inv_z; pv[6] = b.z * inv_z; pv[7] = b.w * inv_z;
            } else {
              const uint4 x8 = __ldg(vp + i);
              const uint32_t xw[4] = {x8.x, x8.y, x8.z, x8.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                pv[2 * h] = ex2(fmaf(bf16_lo(xw[h]), kLog2e, -bp));
                pv[2 * h + 1] = ex2(fmaf(bf16_hi(xw[h]), kLog2e, -bp));
              }
            }
            const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
            float d[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              d[2 * h] = fmaxf(0.f, pv[2 * h] - ex2(fmaf(bf16_lo(yw[h]), kLog2e, -bq)));
              d[2 * h + 1] = fmaxf(0.f, pv[2 * h + 1] - ex2(fmaf(bf16_hi(yw[h]), kLog2e, -bq)));
            }
            bo[2 * i] = make_float4(d[0], d[1], d[2], d[3]);
            bo[2 * i + 1] = make_float4(d[4], d[5], d[6], d[7]);
            z += ((d[0] + d[1]) + (d[2] + d[3])) + ((d[4] + d[5]) + (d[6] + d[7]));
          }
          w0 = v0 + nv * 8 + tid;
        }
      }
      for (int w = w0; w < v1; w += kRsThreads) {
        const float pv = resid ? buf[w] * inv_z : ex2(fmaf(rs_val(prow, w), kLog2e, -bp));
        const float qv = ex2(fmaf(rs_val(qrow, w), kLog2e, -bq));
        const float d = fmaxf(0.f, pv - qv);
        buf[w] = d;
        z += d;
      }
      const float zc = rs_cta_sum0(sh, z);
      rs_exchange(sh, e++, zc, 0.f, 0.f, 0.f);   // (its cluster barrier also publishes buf)
      if (tid == 0) {
        float Z = 0.f;
        for (int k = 0; k < kRsCluster; ++k) Z += sh.all[k][0];
        sh.res[2] = Z > 0.f ? 1.f / Z : 0.f;
      }
      __syncthreads();
      if (sh.res[2] > 0.f) {
        resid = true;
        inv_z = sh.res[2];
      } else {
        resid = false;   // degenerate (rounding only): back to the target softmax
      }
    }
    if (next < 0) {
      // bonus token: the smallest j with cumulative p'(<= j) > u * total.
      // Warp w of each CTA sums a contiguous eighth of the slice (coalesced),
      // the slice totals are exchanged, and in the CTA and warp whose range
      // holds the target the warp walks its range 32 tokens at a time.
      auto pval = [&](int j) -> float {
        return resid ? buf[j] : ex2(fmaf(rs_val(prow, j), kLog2e, -bp));
      };
      const int wlen = (v1 - v0 + kRsWarps - 1) / kRsWarps;
      const int c0 = min(v1, v0 + warp * wlen), c1 = min(v1, c0 + wlen);
      float part = 0.f;
      for (int j = c0 + lane; j < c1; j += 32) part += pval(j);
      part = warp_sum(part);
      if (lane == 0) sh.wred[warp][2] = part;
      __syncthreads();
      float ctot = 0.f;
      if (tid == 0)
        for (int w = 0; w < kRsWarps; ++w) ctot += sh.wred[w][2];
      rs_exchange(sh, e++, ctot, 0.f, 0.f, 0.f);
      if (tid == 0) {   // the owning slice (the first whose range holds the target), and the target in it
        float total = 0.f;
        for (int k = 0; k < kRsCluster; ++k) total += sh.all[k][0];
        const float target = u_final[r] * total;
        int own = -1;
        float lo = 0.f, own_lo = 0.f;
        for (int k = 0; k < kRsCluster; ++k) {
          const float t = sh.all[k][0];
          if (own < 0 && t > 0.f && lo <= target && target < lo + t) { own = k; own_lo = lo; }
          lo += t;
        }
        sh.res[3] = target - own_lo;
        sh.own = own;
        sh.pick = INT32_MAX;
      }
      __syncthreads();
      const int owner = sh.own;
      if (owner == static_cast<int>(rank)) {
        const float target = sh.res[3];
        float lo = 0.f;
        for (int w = 0; w < warp; ++w) lo += sh.wred[w][2];
        const float mine = sh.wred[warp][2];
        // the first warp whose range holds the target (a later one only by rounding)
        bool holds = mine > 0.f && lo <= target && target < lo + mine;
        if (holds) {
          float cum = lo;
          int j = c1 - 1;
          for (int b0 = c0; b0 < c1; b0 += 32) {
            const int jj = b0 + lane;
            const float x = jj < c1 ? pval(jj) : 0.f;
            float inc = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, inc, o);
              if (lane >= o) inc += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, jj < c1 && cum + inc > target);
            if (hit) { j = b0 + __ffs(hit) - 1; break; }
            cum += __shfl_sync(0xffffffffu, inc, 31);
          }
          if (lane == 0) atomicMin(&sh.pick, j);   // smallest j among holding warps
        }
        __syncthreads();
        if (tid == 0) bonus[r] = sh.pick == INT32_MAX ? v1 - 1 : sh.pick;
      } else if (owner < 0 && rank == 0 && tid == 0) {
        bonus[r] = V - 1;
      }
      if (rank == 0 && tid == 0) {
        accept_len[r] = depth;
        best_node[r] = cur;
      }
      rs_cluster_sync();   // no CTA leaves while another may still read its shared memory
      return;
    }
    cur = next;
    ++depth;
    if (rank == 0 && tid == 0 && depth <= max_depth) path[static_cast<int64_t>(r) * (max_depth + 1) + depth] = cur;
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
    return tv::launch_pdl(tv::rejection_kernel<uint16_t>, dim3(B * tv::kRsCluster), dim3(tv::kRsThreads), 0, st,
                          parent, tok,
                          static_cast<const uint16_t*>(p_logits), static_cast<const uint16_t*>(q_logits), V, ld,
                          node_off, max_depth, u_node, u_final, accept_len, best_node, path, bonus, buf,
                          tv::aligned(p_logits, 16) && tv::aligned(q_logits, 16) && ld % 8 == 0);
  return tv::launch_pdl(tv::rejection_kernel<float>, dim3(B * tv::kRsCluster), dim3(tv::kRsThreads), 0, st,
                        parent, tok,
                        static_cast<const float*>(p_logits), static_cast<const float*>(q_logits), V, ld, node_off,
                        max_depth, u_node, u_final, accept_len, best_node, path, bonus, buf, false);
}
