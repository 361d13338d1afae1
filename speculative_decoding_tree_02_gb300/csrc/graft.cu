// Graft's on-GPU successor table (Graft page §2 second/third gears, §6):
//   graft_adj_update  rows of verified tokens <- the target's top-k (last wins)
//   graft_retrieve    stage-template expansion from the current token
#include "tv_common.cuh"

namespace tv {

// ---------------------------------------------------------------------------
// graft_adj_update — deterministic "last writer wins".
//
// Up to TV_ADJ_SCAN_MAX nodes (a verification step): CTA b owns table rows
// [b*R, b*R + R).  Its 8 warps split the node list into 8 contiguous, ordered
// segments.  A warp walks its segment 32 nodes at a time; lanes whose tokens
// fall in the CTA's rows group equal tokens with __match_any_sync and only the
// highest lane (the latest node) records its index in the warp's own
// shared-memory row map.  Program order within the warp makes later iterations
// overwrite earlier ones.  After a barrier the thread of row t (each thread
// takes every 256th row) takes the map entry of the last warp that saw t — the
// last node in global order — and copies that node's top-k into the row.
// Eight warps rather than 32: the CTAs (32 KB of row maps instead of 128 KB)
// are placed beside the attention kernel's in a verification step, which took
// the D-cut step from 139.7 to 138.4 us (two warps: 147.6 us, the scan then
// being too long; four: 139.7 us).
// ---------------------------------------------------------------------------
constexpr int kAdjRows = 1024;
constexpr int kAdjWarps = 8;

__global__ void __launch_bounds__(kAdjWarps * 32) adj_update_kernel(
    int32_t* __restrict__ adj, int V, int k, const int32_t* __restrict__ tok,
    const int32_t* __restrict__ topk, int topk_ld, const uint8_t* __restrict__ valid, int n,
    int32_t* __restrict__ n_bad, bool vec4) {
  extern __shared__ int32_t s_win[];   // [kAdjWarps][kAdjRows]
  __shared__ int s_bad[kAdjWarps];
  griddep_wait();
  griddep_release();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kAdjRows;
  int32_t* my = s_win + warp * kAdjRows;
  for (int q = lane; q < kAdjRows; q += 32) my[q] = -1;
  __syncwarp();

  const int seg = (n + kAdjWarps - 1) / kAdjWarps;
  const int beg = warp * seg;
  const int end = min(n, beg + seg);
  int bad = 0;
  for (int i0 = beg; i0 < end; i0 += 32) {
    const int i = i0 + lane;
    int key = -1 - lane;   // unique sentinel: lanes without a row never group
    if (i < end && (!valid || valid[i])) {
      const int t = tok[i];
      if (t < 0 || t >= V) ++bad;
      else if (t >= t0 && t < t0 + kAdjRows) key = t - t0;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == 31 - __clz(grp)) my[key] = i;
    __syncwarp();
  }
  if (blockIdx.x == 0) {
    bad = __reduce_add_sync(0xffffffffu, bad);
    if (lane == 0) s_bad[warp] = bad;
  }
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0 && n_bad) {
    int b = 0;
    for (int w = 0; w < kAdjWarps; ++w) b += s_bad[w];
    *n_bad = b;
  }
  for (int row = threadIdx.x; row < kAdjRows && t0 + row < V; row += kAdjWarps * 32) {
    int win = -1;
#pragma unroll
    for (int w = 0; w < kAdjWarps; ++w) {
      const int v = s_win[w * kAdjRows + row];
      win = v >= 0 ? v : win;
    }
    if (win < 0) continue;
    const int32_t* src = topk + static_cast<int64_t>(win) * topk_ld;
    int32_t* dst = adj + static_cast<int64_t>(t0 + row) * k;
    if (vec4) {
      for (int c = 0; c < k; c += 4)
        *reinterpret_cast<int4*>(dst + c) = *reinterpret_cast<const int4*>(src + c);
    } else {
      for (int c = 0; c < k; ++c) dst[c] = src[c];
    }
  }
}

// Large batches (n > TV_ADJ_SCAN_MAX, e.g. a whole-table refresh): the scan
// above would read the node list once per table slice.  Instead: last[t] =
// largest valid node index with token t (integer atomicMax: the same result
// in any order), then one thread per row copies the winner's top-k.
__global__ void __launch_bounds__(256) adj_last_init_kernel(int32_t* __restrict__ last, int V,
                                                            int32_t* __restrict__ n_bad) {
  griddep_wait();
  griddep_release();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < V) last[t] = -1;
  if (t == 0 && n_bad) *n_bad = 0;
}

__global__ void __launch_bounds__(256) adj_last_kernel(int32_t* __restrict__ last, int V,
                                                       const int32_t* __restrict__ tok,
                                                       const uint8_t* __restrict__ valid, int n,
                                                       int32_t* __restrict__ n_bad) {
  griddep_wait();
  griddep_release();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  bool bad = false;
  if (i < n && (!valid || valid[i])) {
    const int t = tok[i];
    if (t < 0 || t >= V) bad = true;
    else atomicMax(&last[t], i);
  }
  const unsigned b = __ballot_sync(0xffffffffu, bad);
  if (b && (threadIdx.x & 31) == 0 && n_bad) atomicAdd(n_bad, __popc(b));
}

__global__ void __launch_bounds__(256) adj_copy_kernel(int32_t* __restrict__ adj, int V, int k,
                                                       const int32_t* __restrict__ last,
                                                       const int32_t* __restrict__ topk, int topk_ld,
                                                       bool vec4) {
  griddep_wait();
  griddep_release();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= V) return;
  const int win = last[t];
  if (win < 0) return;
  const int32_t* src = topk + static_cast<int64_t>(win) * topk_ld;
  int32_t* dst = adj + static_cast<int64_t>(t) * k;
  if (vec4) {
    for (int c = 0; c < k; c += 4)
      *reinterpret_cast<int4*>(dst + c) = *reinterpret_cast<const int4*>(src + c);
  } else {
    for (int c = 0; c < k; ++c) dst[c] = src[c];
  }
}

// ---------------------------------------------------------------------------
// graft_retrieve — one thread per (request, slot).  The thread collects the
// ranks on its slot's template path (walking tparent up to the root token)
// and replays them down through the table, so no slot waits for another;
// each lookup is one row/column fetch (Graft page §2: the table lookup is a
// single matrix element read).
// ---------------------------------------------------------------------------
constexpr int kMaxTemplateDepth = 64;

__global__ void __launch_bounds__(128) retrieve_kernel(
    const int32_t* __restrict__ adj, int V, int k, const int32_t* __restrict__ root_tok,
    const int32_t* __restrict__ stage, int B, const int32_t* __restrict__ tparent,
    const int32_t* __restrict__ trank, const int32_t* __restrict__ tmpl_off, int n_stage,
    int max_slots, int32_t* __restrict__ rtok, int32_t* __restrict__ rparent,
    int32_t* __restrict__ nslots, int32_t* __restrict__ err) {
  griddep_wait();
  griddep_release();
  const int b = blockIdx.y;
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B || s >= max_slots) return;
  const int st = stage[b];
  int S = 0, s0 = 0;
  bool bad = false;
  if (st >= 0 && st < n_stage) {
    s0 = tmpl_off[st];
    S = tmpl_off[st + 1] - s0;
    if (S < 0) { S = 0; bad = true; }
    if (S > max_slots) { S = max_slots; bad = true; }
  } else {
    bad = true;
  }
  if (s == 0) nslots[b] = S;
  const int64_t o = static_cast<int64_t>(b) * max_slots + s;
  if (s >= S) {
    rtok[o] = -1;
    rparent[o] = -1;
    if (bad && s == 0 && err) *err = 1;
    return;
  }
  int ranks[kMaxTemplateDepth];
  int depth = 0;
  int j = s;
  while (j >= 0) {
    const int p = tparent[s0 + j];
    const int r = trank[s0 + j];
    if (depth == kMaxTemplateDepth || p >= j || p < -1 || r < 0 || r >= k) { bad = true; break; }
    ranks[depth++] = r;
    j = p;
  }
  int t = root_tok[b];
  if (!bad) {
    for (int d = depth - 1; d >= 0; --d) {
      if (t < 0 || t >= V) { bad = true; break; }
      t = adj[static_cast<int64_t>(t) * k + ranks[d]];
    }
    if (t < 0 || t >= V) bad = true;
  }
  rtok[o] = bad ? -1 : t;
  rparent[o] = tparent[s0 + s];
  if (bad && err) *err = 1;
}

}  // namespace tv

TV_API size_t graft_adj_update_workspace_size(int V, int n) {
  if (V <= 0 || n <= TV_ADJ_SCAN_MAX) return 0;
  return (static_cast<size_t>(V) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}

TV_API int graft_adj_update(int32_t* adj, int V, int k, const int32_t* tok,
                            const int32_t* topk_idx, int topk_ld, const uint8_t* valid, int n,
                            int32_t* n_bad, void* ws, size_t ws_bytes, tv_stream_t stream) {
  if (V <= 0 || k <= 0 || n < 0 || topk_ld < k) return TV_EINVAL;
  if (k > TV_MAX_TOPK) return TV_EUNSUPPORTED;
  if (n == 0) return TV_OK;
  if (!adj || !tok || !topk_idx) return TV_EINVAL;
  // rows and top-k records start on 16-byte boundaries: copy 4 ints at a time
  const bool vec4 = (k % 4 == 0) && (topk_ld % 4 == 0) && tv::aligned(adj, 16) &&
                    tv::aligned(topk_idx, 16);
  auto st = reinterpret_cast<cudaStream_t>(stream);
  if (n > TV_ADJ_SCAN_MAX) {
    if (!ws || ws_bytes < graft_adj_update_workspace_size(V, n) || !tv::aligned(ws, 16)) return TV_EWORKSPACE;
    auto* last = static_cast<int32_t*>(ws);
    const int gv = (V + 255) / 256, gn = (n + 255) / 256;
    int rc = tv::launch_pdl(tv::adj_last_init_kernel, dim3(gv), dim3(256), 0, st, last, V, n_bad);
    if (rc == TV_OK) rc = tv::launch_pdl(tv::adj_last_kernel, dim3(gn), dim3(256), 0, st, last, V, tok, valid, n, n_bad);
    if (rc == TV_OK)
      rc = tv::launch_pdl(tv::adj_copy_kernel, dim3(gv), dim3(256), 0, st, adj, V, k, last, topk_idx, topk_ld, vec4);
    return rc;
  }
  const int smem = tv::kAdjWarps * tv::kAdjRows * static_cast<int>(sizeof(int32_t));
  if (!tv::smem_limit(tv::adj_update_kernel, smem)) return TV_ECUDA;
  const int grid = (V + tv::kAdjRows - 1) / tv::kAdjRows;
  return tv::launch_pdl(tv::adj_update_kernel, dim3(grid), dim3(tv::kAdjWarps * 32), smem, st, adj, V, k, tok,
                        topk_idx, topk_ld, valid, n, n_bad, vec4);
}

TV_API int graft_retrieve(const int32_t* adj, int V, int k, const int32_t* root_tok,
                          const int32_t* stage, int B, const int32_t* tparent,
                          const int32_t* trank, const int32_t* tmpl_off, int n_stage,
                          int max_slots, int32_t* rtok, int32_t* rparent, int32_t* nslots,
                          int32_t* err, tv_stream_t stream) {
  if (V <= 0 || k <= 0 || B < 0 || n_stage <= 0 || max_slots < 0) return TV_EINVAL;
  if (B == 0 || max_slots == 0) return TV_OK;
  if (!adj || !root_tok || !stage || !tmpl_off || !rtok || !rparent || !nslots) return TV_EINVAL;
  if (!tparent || !trank) return TV_EINVAL;
  if (B > 65535) return TV_EUNSUPPORTED;
  dim3 grid((max_slots + 127) / 128, B);
  return tv::launch_pdl(tv::retrieve_kernel, grid, dim3(128), 0, reinterpret_cast<cudaStream_t>(stream), adj, V, k,
                        root_tok, stage, B, tparent, trank, tmpl_off, n_stage, max_slots, rtok, rparent, nslots,
                        err);
}
