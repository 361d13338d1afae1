// Graft tree planning on the GPU, on either side of the verification step:
//   graft_stage_decide  calibrated pruning checkpoints (Graft page §2, first
//                       gear): best cumulative confidence at draft layers
//                       0, 1, 5 against thresholds -> pruning stage
//   graft_replace       batched static-tree variant (§4) and Graft-TAIL (§7):
//                       low-confidence draft nodes are replaced by retrieval
//                       nodes from the successor table, slot count fixed
// One CTA per request, one thread per node.  Cumulative confidences are fp32
// products in root-to-node order, computed one tree level at a time so that
// every product is formed from its parent's finished value.
#include <algorithm>

#include "tv_common.cuh"

namespace tv {

constexpr int kPlanMaxNodes = TV_MAX_NODES;
constexpr int kCheckpoints = 3;
__constant__ int kCheckpointLayer[kCheckpoints] = {0, 1, 5};

struct Taus { float t[kCheckpoints]; };

// Depth (root 0) and cumulative confidence of node i of a request whose n
// nodes are staged in s_par (request-local parents, -1 = root).  Nodes whose
// parent chain is malformed (an index out of range, or longer than n) get
// depth -1 and are left out.  All threads of the CTA call this.
__device__ void tree_levels(const int16_t* s_par, const float* conf_g, int n, int* s_depth, float* s_c,
                            int* s_maxd, bool* bad) {
  const int i = threadIdx.x;
  int d = -1;
  if (i < n) {
    int p = s_par[i], steps = 0;
    while (p >= 0 && p < n && steps <= n) { p = s_par[p]; ++steps; }
    d = (p == -1 && steps <= n) ? steps : -1;
    if (s_par[i] >= n || s_par[i] < -1) d = -1;
    s_depth[i] = d;
    s_c[i] = 1.f;
  }
  if (threadIdx.x == 0) *s_maxd = 0;
  __syncthreads();
  if (i < n) {
    if (d < 0) *bad = true;
    else atomicMax(s_maxd, d);
  }
  __syncthreads();
  const int maxd = *s_maxd;
  for (int L = 1; L <= maxd; ++L) {
    if (i < n && d == L) s_c[i] = __fmul_rn(s_c[s_par[i]], conf_g[i]);
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024) stage_decide_kernel(const int32_t* __restrict__ parent,
                                                            const float* __restrict__ conf,
                                                            const int32_t* __restrict__ node_off, Taus tau,
                                                            int32_t* __restrict__ stage, float* __restrict__ best,
                                                            int32_t* __restrict__ err) {
  __shared__ int16_t s_par[kPlanMaxNodes];
  __shared__ int s_depth[kPlanMaxNodes];
  __shared__ float s_c[kPlanMaxNodes];
  __shared__ float s_best[kCheckpoints][32];
  __shared__ int s_maxd;
  __shared__ bool s_bad;
  griddep_wait();
  griddep_release();
  const int r = blockIdx.x, i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const int n0 = node_off[r];
  const int n = min(node_off[r + 1] - n0, kPlanMaxNodes);
  if (i == 0) s_bad = false;
  if (i < n) s_par[i] = static_cast<int16_t>(max(-2, min(parent[n0 + i], kPlanMaxNodes)));
  __syncthreads();
  tree_levels(s_par, conf + n0, n, s_depth, s_c, &s_maxd, &s_bad);
  // best cumulative confidence per checkpoint layer (a layer without nodes: 0)
  float b[kCheckpoints];
#pragma unroll
  for (int j = 0; j < kCheckpoints; ++j) {
    b[j] = (i < n && s_depth[i] == kCheckpointLayer[j] + 1) ? s_c[i] : 0.f;
    b[j] = warp_max(b[j]);
    if (lane == 0) s_best[j][warp] = b[j];
  }
  __syncthreads();
  if (i == 0) {
    int st = kCheckpoints;
    for (int j = 0; j < kCheckpoints; ++j) {
      float m = 0.f;
      for (int w = 0; w < (blockDim.x + 31) / 32; ++w) m = fmaxf(m, s_best[j][w]);
      if (best) best[r * kCheckpoints + j] = m;
      if (st == kCheckpoints && m < tau.t[j]) st = j;
    }
    stage[r] = st;
    if (s_bad && err) atomicExch(err, 1);
  }
}

// Request r's tree is nodes r*S .. r*S+S-1 (node 0 of each is its root).
__global__ void __launch_bounds__(1024) replace_kernel(
    const int32_t* __restrict__ parent, const int32_t* __restrict__ tok, const float* __restrict__ conf, int S,
    float tau, int attach, const int32_t* __restrict__ adj, int V, int k, const int32_t* __restrict__ tparent,
    const int32_t* __restrict__ trank, int n_tmpl, int32_t* __restrict__ tok_out, int32_t* __restrict__ par_out,
    int32_t* __restrict__ n_kept, int32_t* __restrict__ err) {
  __shared__ int16_t s_par[kPlanMaxNodes];
  __shared__ int s_depth[kPlanMaxNodes];
  __shared__ float s_c[kPlanMaxNodes];
  __shared__ uint8_t s_keep[kPlanMaxNodes];
  __shared__ int s_new[kPlanMaxNodes];
  __shared__ int s_w[32];
  __shared__ unsigned long long s_anchor;
  __shared__ int s_maxd;
  __shared__ bool s_bad;
  griddep_wait();
  griddep_release();
  const int r = blockIdx.x, i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const int n0 = r * S;
  if (i == 0) { s_bad = false; s_anchor = 0ull; }
  if (i < S) {
    s_par[i] = static_cast<int16_t>(i == 0 ? -1 : max(-2, min(parent[n0 + i], kPlanMaxNodes)));
    s_keep[i] = 0;
  }
  __syncthreads();
  tree_levels(s_par, conf + n0, S, s_depth, s_c, &s_maxd, &s_bad);
  // keep: the whole path clears the threshold (one level at a time)
  if (i == 0) s_keep[0] = 1;
  __syncthreads();
  for (int L = 1; L <= s_maxd; ++L) {
    if (i < S && s_depth[i] == L) s_keep[i] = s_c[i] >= tau && s_keep[s_par[i]];
    __syncthreads();
  }
  // compaction: exclusive scan of the keep flags in node order
  const int f = i < S ? s_keep[i] : 0;
  int x = f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) / 32;
    const int w = lane < nw ? s_w[lane] : 0;
    int iw = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, iw, o);
      if (lane >= o) iw += y;
    }
    if (lane < nw) s_w[lane] = iw - w;
    if (lane == 31) s_maxd = iw;                  // total kept (s_maxd is free again)
  }
  __syncthreads();
  const int nk = s_maxd;
  const int mine = s_w[warp] + x - f;
  if (i < S) s_new[i] = f ? mine : -1;
  // anchor of the retrieval subtree: root, or the deepest kept node (then the
  // larger cumulative confidence, then the lower index)
  if (attach == 1 && f) {
    const unsigned long long key = (static_cast<unsigned long long>(s_depth[i]) << 53) |
                                   (static_cast<unsigned long long>(__float_as_uint(s_c[i])) << 21) |
                                   static_cast<unsigned long long>((1 << 21) - 1 - i);
    atomicMax(&s_anchor, key);
  }
  __syncthreads();
  const int anchor = attach == 1 ? (1 << 21) - 1 - static_cast<int>(s_anchor & ((1ull << 21) - 1)) : 0;
  if (f) {
    const int p = s_par[i];
    tok_out[n0 + mine] = tok[n0 + i];
    par_out[n0 + mine] = i == 0 ? -1 : s_new[p];
  }
  __syncthreads();
  // retrieval slots: slot s replays its template path down from the anchor
  const int F = min(S - nk, n_tmpl);
  const int atok = tok[n0 + anchor];
  for (int s = i; s < S - nk; s += blockDim.x) {
    int out_tok = -1, out_par = -1;
    if (s < F) {
      int ranks[64], d = 0, t = s;
      bool ok = true;
      while (t >= 0 && d < 64) {
        if (t >= n_tmpl || trank[t] < 0 || trank[t] >= k) { ok = false; break; }
        ranks[d++] = trank[t];
        const int tp = tparent[t];
        if (tp >= t) { ok = false; break; }
        t = tp;
      }
      ok = ok && t < 0;
      int src = atok;
      for (int q = d - 1; ok && q >= 0; --q) {
        if (src < 0 || src >= V) { ok = false; break; }
        src = adj[static_cast<int64_t>(src) * k + ranks[q]];
      }
      if (ok && (src < 0 || src >= V)) ok = false;
      if (ok) {
        out_tok = src;
        const int tp = tparent[s];
        out_par = tp < 0 ? s_new[anchor] : nk + tp;
      } else if (err) {
        atomicExch(err, 1);
      }
    }
    tok_out[n0 + nk + s] = out_tok;
    par_out[n0 + nk + s] = out_par;
  }
  if (i == 0) {
    n_kept[r] = nk;
    if (s_bad && err) atomicExch(err, 1);
  }
}

}  // namespace tv

TV_API int graft_stage_decide(const int32_t* parent, const float* conf, const int32_t* node_off, int B,
                              int max_nodes, const float* tau, int32_t* stage, float* best, int32_t* err,
                              tv_stream_t stream) {
  if (B < 0 || max_nodes < 0) return TV_EINVAL;
  if (max_nodes > TV_MAX_NODES) return TV_EUNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!parent || !conf || !node_off || !tau || !stage) return TV_EINVAL;
  tv::Taus t{};
  for (int j = 0; j < tv::kCheckpoints; ++j) {
    if (!(tau[j] >= 0.f)) return TV_EINVAL;   // host array; NaN rejected
    t.t[j] = tau[j];
  }
  const int threads = std::max(32, (max_nodes + 31) / 32 * 32);
  return tv::launch_pdl(tv::stage_decide_kernel, dim3(B), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream),
                        parent, conf, node_off, t, stage, best, err);
}

TV_API int graft_replace(const int32_t* parent, const int32_t* tok, const float* conf, int B, int S, float tau,
                         int attach, const int32_t* adj, int V, int k, const int32_t* tparent,
                         const int32_t* trank, int n_tmpl, int32_t* tok_out, int32_t* parent_out,
                         int32_t* n_kept, int32_t* err, tv_stream_t stream) {
  if (B < 0 || S < 0 || V <= 0 || k <= 0 || n_tmpl < 0) return TV_EINVAL;
  if (attach != 0 && attach != 1) return TV_EINVAL;
  if (!(tau == tau)) return TV_EINVAL;
  if (S > TV_MAX_NODES || k > TV_MAX_TOPK) return TV_EUNSUPPORTED;
  if (B == 0 || S == 0) return TV_OK;
  if (!parent || !tok || !conf || !adj || !tok_out || !parent_out || !n_kept) return TV_EINVAL;
  if (n_tmpl > 0 && (!tparent || !trank)) return TV_EINVAL;
  const int threads = std::max(32, (S + 31) / 32 * 32);
  return tv::launch_pdl(tv::replace_kernel, dim3(B), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream),
                        parent, tok, conf, S, tau, attach, adj, V, k, tparent, trank, n_tmpl, tok_out, parent_out,
                        n_kept, err);
}
