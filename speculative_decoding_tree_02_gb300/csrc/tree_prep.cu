// tv_tree_prep: depth, position ids, ancestor bitmask and visible prefix of a
// flattened candidate tree (Graft page §2 third gear; SpecOPD page §02 mask).
//
// One thread per (node, ancestor word): the thread walks the node's parent
// chain and sets the bits that fall into its 64-node word, so each u64 of the
// [n, W] mask is produced by exactly one thread with one coalesced store.
#include "tv_common.cuh"

namespace tv {

__global__ void __launch_bounds__(256) tree_prep_kernel(
    const int32_t* __restrict__ parent, const int32_t* __restrict__ node_off,
    const int32_t* __restrict__ prefix_len, const int32_t* __restrict__ vis_prefix, int W,
    int32_t* __restrict__ depth, int32_t* __restrict__ pos, uint64_t* __restrict__ anc,
    int32_t* __restrict__ vis_out, int32_t* __restrict__ err) {
  griddep_wait();
  griddep_release();
  const int r = blockIdx.y;
  const int n0 = node_off[r];
  const int N = node_off[r + 1] - n0;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = t / W;
  const int w = t - i * W;
  if (i >= N) return;
  const int lo = w * 64;
  uint64_t bits = 0;
  int d = 0;
  bool bad = false;
  int j = i;
  // Walk to the root.  Each valid step strictly decreases j, so at most i
  // steps; an index outside [-1, j) ends the walk and is reported.
  for (int steps = 0; steps <= i; ++steps) {
    if (j >= lo && j < lo + 64) bits |= 1ull << (j - lo);
    const int p = parent[n0 + j];
    if (p < 0) {
      if (p != -1) bad = true;
      break;
    }
    if (p >= j) {
      bad = true;
      break;
    }
    j = p;
    ++d;
  }
  anc[static_cast<int64_t>(n0 + i) * W + w] = bits;
  if (w == 0) {
    const int P = prefix_len[r];
    int v = vis_prefix ? vis_prefix[n0 + i] : P;
    v = v < 0 ? 0 : (v > P ? P : v);
    depth[n0 + i] = d;
    pos[n0 + i] = v + d;
    vis_out[n0 + i] = v;
    if (bad && err) *err = 1;
  }
}

}  // namespace tv

TV_API int tv_tree_prep(const int32_t* parent, const int32_t* node_off, const int32_t* prefix_len,
                        const int32_t* vis_prefix, int B, int max_nodes, int anc_words,
                        int32_t* depth, int32_t* pos, uint64_t* anc, int32_t* vis_out,
                        int32_t* err, tv_stream_t stream) {
  if (B < 0 || max_nodes < 0 || anc_words < 1) return TV_EINVAL;
  if (max_nodes > TV_MAX_NODES) return TV_EUNSUPPORTED;
  if (anc_words < (max_nodes + 63) / 64) return TV_EINVAL;
  if (B == 0 || max_nodes == 0) return TV_OK;
  if (!parent || !node_off || !prefix_len || !depth || !pos || !anc || !vis_out) return TV_EINVAL;
  if (B > 65535) return TV_EUNSUPPORTED;
  const int per_req = max_nodes * anc_words;
  dim3 grid((per_req + 255) / 256, B);
  return tv::launch_pdl(tv::tree_prep_kernel, grid, dim3(256), 0, reinterpret_cast<cudaStream_t>(stream), parent,
                        node_off, prefix_len, vis_prefix, anc_words, depth, pos, anc, vis_out, err);
}
