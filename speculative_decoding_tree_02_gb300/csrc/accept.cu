// accept_longest_path: greedy longest accepted path per request (Graft page
// §2 third gear; BlockPilot page intro; SpecOPD page §01 and §03 example).
//
// One CTA per request, one thread per node.  The tree (parents, match flags)
// is staged in shared memory; each thread walks its own root path twice (once
// for its depth, once to find the first rejected step), so no thread waits
// on another.  The deepest accepted node (lowest index on ties) is found with
// a block max over a packed (depth, -index) key.
#include "tv_common.cuh"

namespace tv {

__global__ void __launch_bounds__(1024) accept_kernel(
    const int32_t* __restrict__ parent, const int32_t* __restrict__ tok,
    const int32_t* __restrict__ argmax, const uint8_t* __restrict__ valid,
    const int32_t* __restrict__ node_off, int max_depth, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ best_node, int32_t* __restrict__ path, int32_t* __restrict__ bonus,
    int32_t* __restrict__ path_acc) {
  __shared__ int16_t s_par[TV_MAX_NODES];
  __shared__ uint8_t s_ok[TV_MAX_NODES];
  __shared__ int16_t s_path[TV_MAX_NODES];
  __shared__ int s_warp_best[32];
  __shared__ int s_best;

  griddep_wait();
  griddep_release();
  const int r = blockIdx.x;
  const int n0 = node_off[r];
  const int N = min(node_off[r + 1] - n0, TV_MAX_NODES);
  const int i = threadIdx.x;

  // ok(i): the node passes its own check (valid, and for a non-root its token
  // equals the target's argmax at its parent).  Out-of-range parents make a
  // node a root, matching tv_tree_prep.
  if (i < N) {
    int p = parent[n0 + i];
    if (p >= i || p < -1) p = -1;
    s_par[i] = static_cast<int16_t>(p);
    bool ok = valid ? valid[n0 + i] != 0 : true;
    if (ok && p >= 0) ok = tok[n0 + i] == argmax[n0 + p];
    s_ok[i] = ok;
  }
  __syncthreads();

  int key = -1;
  if (i < N) {
    int d = 0;
    for (int j = s_par[i]; j >= 0; j = s_par[j]) ++d;
    // first failing depth on root..i (d+1 when none)
    int first_bad = d + 1;
    int t = d;
    for (int j = i; j >= 0; j = s_par[j], --t)
      if (!s_ok[j]) first_bad = t;
    const int pa = first_bad - 1;
    if (path_acc) path_acc[n0 + i] = pa;
    if (pa == d) key = (d << 11) | (2047 - i);
  }
  key = warp_max(key);
  if ((threadIdx.x & 31) == 0) s_warp_best[threadIdx.x >> 5] = key;
  __syncthreads();
  if (threadIdx.x < 32) {
    int v = threadIdx.x < (blockDim.x + 31) / 32 ? s_warp_best[threadIdx.x] : -1;
    v = warp_max(v);
    if (threadIdx.x == 0) s_best = v;
  }
  __syncthreads();
  const int kbest = s_best;
  const int best = kbest < 0 ? -1 : 2047 - (kbest & 2047);
  const int best_d = kbest < 0 ? -1 : (kbest >> 11);
  if (threadIdx.x == 0) {
    accept_len[r] = best_d;
    best_node[r] = best;
    bonus[r] = best >= 0 ? argmax[n0 + best] : -1;
    int t = best_d;
    for (int j = best; j >= 0; j = s_par[j]) s_path[t--] = static_cast<int16_t>(j);
  }
  __syncthreads();
  for (int t = threadIdx.x; t <= max_depth; t += blockDim.x)
    path[static_cast<int64_t>(r) * (max_depth + 1) + t] = t <= best_d ? s_path[t] : -1;
}

}  // namespace tv

TV_API int accept_longest_path(const int32_t* parent, const int32_t* tok, const int32_t* argmax,
                               const uint8_t* valid, const int32_t* node_off, int B, int max_nodes,
                               int max_depth, int32_t* accept_len, int32_t* best_node,
                               int32_t* path, int32_t* bonus, int32_t* path_acc,
                               tv_stream_t stream) {
  if (B < 0 || max_nodes < 0 || max_depth < 0) return TV_EINVAL;
  if (max_nodes > TV_MAX_NODES) return TV_EUNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!parent || !tok || !argmax || !node_off || !accept_len || !best_node || !path || !bonus)
    return TV_EINVAL;
  if (B > (1 << 30)) return TV_EUNSUPPORTED;
  const int threads = max(32, (max_nodes + 31) / 32 * 32);
  return tv::launch_pdl(tv::accept_kernel, dim3(B), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream),
                        parent, tok, argmax, valid, node_off, max_depth, accept_len, best_node, path, bonus,
                        path_acc);
}
