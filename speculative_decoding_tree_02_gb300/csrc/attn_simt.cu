// tree_verify_attn, SIMT path: tree-masked grouped-query attention of the
// candidate nodes over a shared KV prefix (Graft page §2 third gear; SpecOPD
// page §02 proposal-tree scoring with the ancestor mask).
//
// Work unit (CTA): one request, one KV head, a tile of query rows and one
// split of the prefix keys.  The tile holds 64 query rows = (nodes x g heads
// that share the KV head), 4 threads per row (each owns d/4 dims of q and of
// the output accumulator).  Keys stream through shared memory 32 at a time,
// first the CTA's split of the visible prefix, then (last split only) the
// range of tree nodes that can be ancestors of the tile's nodes.  Visibility
// is decided in registers: prefix key kp is visible iff kp < vis(node), tree
// key j iff bit j of the node's ancestor row is set.  Online softmax in base
// 2 with fp32 accumulation.  With several splits, each writes a normalised
// partial (o, m, l) and a combine kernel merges them in split order.
#include <cmath>

#include "attn.cuh"

namespace tv {

constexpr int kSRows = 64;          // query rows per CTA
constexpr int kSTpr = 4;            // threads per row
constexpr int kSThreads = kSRows * kSTpr;
constexpr int kSTk = 32;            // keys per shared-memory tile

template <typename T, int D>
__device__ __forceinline__ void load_key_row(const T* src, float* dst, int tid_in_row, int lanes) {
  // D elements of one key row into fp32 shared memory; `lanes` threads cooperate
  if constexpr (sizeof(T) == 2) {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
    for (int c = tid_in_row; c < D / 8; c += lanes) {
      uint4 w = *reinterpret_cast<const uint4*>(s + c * 8);
      float4 a = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
      float4 b = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
      *reinterpret_cast<float4*>(dst + c * 8) = a;
      *reinterpret_cast<float4*>(dst + c * 8 + 4) = b;
    }
  } else {
    const float* s = reinterpret_cast<const float*>(src);
    for (int c = tid_in_row; c < D / 4; c += lanes)
      *reinterpret_cast<float4*>(dst + c * 4) = *reinterpret_cast<const float4*>(s + c * 4);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kSThreads, 2) attn_simt_kernel(AttnParams p) {
  constexpr int DPT = D / kSTpr;     // dims per thread
  constexpr int NV = DPT / 4;        // float4 groups per thread
  __shared__ __align__(16) float s_k[kSTk][D];
  __shared__ __align__(16) float s_v[kSTk][D];
  __shared__ int s_red[kSThreads / 32][3];

  const int tid = threadIdx.x;
  const int row = tid / kSTpr, part = tid % kSTpr;
  const int split = blockIdx.x, tile = blockIdx.y;
  const int r = blockIdx.z / p.Hkv, kvh = blockIdx.z % p.Hkv;
  const int g = p.Hq / p.Hkv;
  const int nq = kSRows / g;                      // nodes per tile
  const int n0 = p.node_off[r];
  const int N = p.node_off[r + 1] - n0;
  // rows past max_nodes have no workspace slot: the caller's bound is enforced
  const int cnt = min(p.node_cnt ? min(p.node_cnt[r], N) : N, p.max_nodes);
  const int node_first = tile * nq;
  if (node_first >= cnt) return;                  // whole CTA idle (uniform)
  const int pre0 = p.pre_off[r];
  const int P = p.pre_off[r + 1] - pre0;

  const int ln = node_first + row / g;             // request-local node of this row
  const int head = kvh * g + row % g;
  const bool active = (row < nq * g) && ln < cnt;
  const int gn = n0 + ln;                          // global node index

  int vis = 0, lowest = 1 << 30;
  if (active) {
    vis = p.vis_prefix ? p.vis_prefix[gn] : P;
    vis = min(max(vis, 0), P);
    for (int w = 0; w < p.anc_words; ++w) {
      const uint64_t a = p.anc[static_cast<int64_t>(gn) * p.anc_words + w];
      if (a) { lowest = w * 64 + __ffsll(static_cast<long long>(a)) - 1; break; }
    }
  }
  // CTA-wide: prefix extent and tree-key range
  {
    int vmax = __reduce_max_sync(0xffffffffu, vis);
    int lmin = __reduce_min_sync(0xffffffffu, lowest);
    int hmax = __reduce_max_sync(0xffffffffu, active ? ln : -1);
    if ((tid & 31) == 0) { s_red[tid >> 5][0] = vmax; s_red[tid >> 5][1] = lmin; s_red[tid >> 5][2] = hmax; }
  }
  __syncthreads();
  int vmax = 0, tlo = 1 << 30, thi = -1;
  for (int w = 0; w < kSThreads / 32; ++w) {
    vmax = max(vmax, s_red[w][0]);
    tlo = min(tlo, s_red[w][1]);
    thi = max(thi, s_red[w][2]);
  }

  // q (pre-scaled into base-2 logits) and accumulators
  const float qs = p.scale * kLog2e;
  float q[DPT], o[DPT];
  if (active) {
    const T* qp = static_cast<const T*>(p.q) + (static_cast<int64_t>(gn) * p.Hq + head) * D;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int d0 = 16 * i + 4 * part;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x;
        if constexpr (sizeof(T) == 2) x = bf16_at(reinterpret_cast<const uint16_t*>(qp) + d0 + e);
        else x = reinterpret_cast<const float*>(qp)[d0 + e];
        q[4 * i + e] = x * qs;
      }
    }
  } else {
#pragma unroll
    for (int t = 0; t < DPT; ++t) q[t] = 0.f;
  }
#pragma unroll
  for (int t = 0; t < DPT; ++t) o[t] = 0.f;
  float m = -INFINITY, l = 0.f;

  // key ranges of this CTA
  const int chunk = (p.max_prefix + p.n_split - 1) / p.n_split;
  const int kb = split * chunk;
  const int ke = min(kb + chunk, vmax);
  const bool do_tree = (split == p.n_split - 1) && thi >= 0;
  const int tb = do_tree ? (tlo & ~(kSTk - 1)) : 0;
  const int n_pre_tiles = ke > kb ? (ke - kb + kSTk - 1) / kSTk : 0;
  const int n_tree_tiles = do_tree ? (thi - tb) / kSTk + 1 : 0;
  const T* kpre = static_cast<const T*>(p.k_pre);
  const T* vpre = static_cast<const T*>(p.v_pre);
  const T* ktree = static_cast<const T*>(p.k_tree);
  const T* vtree = static_cast<const T*>(p.v_tree);

  for (int it = 0; it < n_pre_tiles + n_tree_tiles; ++it) {
    const bool tree = it >= n_pre_tiles;
    const int key0 = tree ? tb + (it - n_pre_tiles) * kSTk : kb + it * kSTk;
    const int key_end = tree ? thi + 1 : ke;   // exclusive
    __syncthreads();   // previous tile consumed
    {
      // 256 threads: 8 per key row
      const int j = tid / 8, c = tid % 8;
      const int key = key0 + j;
      float* dk = s_k[j];
      float* dv = s_v[j];
      if (key < key_end) {
        const int64_t rowi = tree ? static_cast<int64_t>(n0 + key) : static_cast<int64_t>(pre0 + key);
        const int64_t off = (rowi * p.Hkv + kvh) * D;
        load_key_row<T, D>((tree ? ktree : kpre) + off, dk, c, 8);
        load_key_row<T, D>((tree ? vtree : vpre) + off, dv, c, 8);
      } else {
        for (int e = c; e < D; e += 8) { dk[e] = 0.f; dv[e] = 0.f; }
      }
    }
    __syncthreads();

    // visibility bits of the 32 keys for this row
    uint32_t vis_bits = 0;
    if (active) {
      if (tree) {
        const int w = key0 >> 6;
        if (w < p.anc_words) {
          const uint64_t a = p.anc[static_cast<int64_t>(gn) * p.anc_words + w];
          vis_bits = static_cast<uint32_t>(a >> (key0 & 63));
        }
        const int valid = key_end - key0;
        if (valid < 32) vis_bits &= (1u << valid) - 1u;
      } else {
        const int valid = min(vis, key_end) - key0;
        vis_bits = valid >= 32 ? 0xffffffffu : (valid > 0 ? (1u << valid) - 1u : 0u);
      }
    }

    float s[kSTk];
#pragma unroll
    for (int j = 0; j < kSTk; ++j) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const float4 kk = *reinterpret_cast<const float4*>(&s_k[j][16 * i + 4 * part]);
        acc = fmaf(q[4 * i + 0], kk.x, acc);
        acc = fmaf(q[4 * i + 1], kk.y, acc);
        acc = fmaf(q[4 * i + 2], kk.z, acc);
        acc = fmaf(q[4 * i + 3], kk.w, acc);
      }
      s[j] = acc;
    }
#pragma unroll
    for (int j = 0; j < kSTk; ++j) {
      s[j] += __shfl_xor_sync(0xffffffffu, s[j], 1);
      s[j] += __shfl_xor_sync(0xffffffffu, s[j], 2);
    }
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < kSTk; ++j) {
      s[j] = (vis_bits >> j) & 1u ? s[j] : -INFINITY;
      mt = fmaxf(mt, s[j]);
    }
    const float mn = fmaxf(m, mt);
    if (mn == -INFINITY) continue;   // nothing visible yet for this row
    const float corr = ex2(m - mn);
    float ps = 0.f;
#pragma unroll
    for (int j = 0; j < kSTk; ++j) {
      s[j] = ex2(s[j] - mn);
      ps += s[j];
    }
    l = l * corr + ps;
#pragma unroll
    for (int t = 0; t < DPT; ++t) o[t] *= corr;
#pragma unroll
    for (int j = 0; j < kSTk; ++j) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const float4 vv = *reinterpret_cast<const float4*>(&s_v[j][16 * i + 4 * part]);
        o[4 * i + 0] = fmaf(s[j], vv.x, o[4 * i + 0]);
        o[4 * i + 1] = fmaf(s[j], vv.y, o[4 * i + 1]);
        o[4 * i + 2] = fmaf(s[j], vv.z, o[4 * i + 2]);
        o[4 * i + 3] = fmaf(s[j], vv.w, o[4 * i + 3]);
      }
    }
    m = mn;
  }
  if (!active) return;

  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (p.n_split == 1) {
    T* op = static_cast<T*>(p.out) + (static_cast<int64_t>(gn) * p.Hq + head) * D;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int d0 = 16 * i + 4 * part;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = o[4 * i + e] * inv;
        if constexpr (sizeof(T) == 2) reinterpret_cast<uint16_t*>(op)[d0 + e] = f2bf(x);
        else reinterpret_cast<float*>(op)[d0 + e] = x;
      }
    }
    if (part == 0 && p.lse)
      p.lse[static_cast<int64_t>(gn) * p.Hq + head] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  } else {
    const int64_t slot = (static_cast<int64_t>(split) * p.B * p.max_nodes +
                          static_cast<int64_t>(r) * p.max_nodes + ln) * p.Hq + head;
    float* po = p.ws_o + slot * D;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float4 v4 = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
      *reinterpret_cast<float4*>(po + 16 * i + 4 * part) = v4;
    }
    if (part == 0) p.ws_ml[slot] = make_float2(m, l);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnParams p) {
  // blockIdx.y = request, blockIdx.x = local node; threads over (head, 4-dim group)
  const int r = blockIdx.y, ln = blockIdx.x;
  const int n0 = p.node_off[r];
  const int N = p.node_off[r + 1] - n0;
  const int cnt = min(p.node_cnt ? min(p.node_cnt[r], N) : N, p.max_nodes);
  if (ln >= cnt) return;
  const int gn = n0 + ln;
  const int64_t per_split = static_cast<int64_t>(p.B) * p.max_nodes * p.Hq;
  for (int t = threadIdx.x; t < p.Hq * (D / 4); t += blockDim.x) {
    const int head = t / (D / 4), c = t % (D / 4);
    const int64_t slot0 = (static_cast<int64_t>(r) * p.max_nodes + ln) * p.Hq + head;
    float M = -INFINITY;
    for (int s = 0; s < p.n_split; ++s) M = fmaxf(M, p.ws_ml[s * per_split + slot0].x);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.n_split; ++s) {
      const float2 ml = p.ws_ml[s * per_split + slot0];
      if (ml.y <= 0.f) continue;
      const float w = ml.y * ex2(ml.x - M);
      L += w;
      const float4 v = *reinterpret_cast<const float4*>(p.ws_o + (s * per_split + slot0) * D + 4 * c);
      acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float res[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
    T* op = static_cast<T*>(p.out) + (static_cast<int64_t>(gn) * p.Hq + head) * D + 4 * c;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if constexpr (sizeof(T) == 2) reinterpret_cast<uint16_t*>(op)[e] = f2bf(res[e]);
      else reinterpret_cast<float*>(op)[e] = res[e];
    }
    if (c == 0 && p.lse)
      p.lse[static_cast<int64_t>(gn) * p.Hq + head] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
}

template <typename T, int D>
int attn_simt_launch(const AttnParams& p, cudaStream_t st) {
  const int g = p.Hq / p.Hkv;
  const int nq = kSRows / g;
  const int tiles = (p.max_nodes + nq - 1) / nq;
  dim3 grid(p.n_split, tiles, p.B * p.Hkv);
  attn_simt_kernel<T, D><<<grid, kSThreads, 0, st>>>(p);
  if (p.n_split > 1) return attn_combine(p, st);
  return launch_status();
}

int attn_combine(const AttnParams& p, cudaStream_t st) {
  dim3 g2(p.max_nodes, p.B);
  if (p.dtype == TV_BF16) {
    if (p.d == 128) attn_combine_kernel<uint16_t, 128><<<g2, 256, 0, st>>>(p);
    else attn_combine_kernel<uint16_t, 64><<<g2, 256, 0, st>>>(p);
  } else {
    if (p.d == 128) attn_combine_kernel<float, 128><<<g2, 256, 0, st>>>(p);
    else attn_combine_kernel<float, 64><<<g2, 256, 0, st>>>(p);
  }
  return launch_status();
}

int attn_simt(const AttnParams& p, cudaStream_t st) {
  if (p.dtype == TV_BF16) {
    if (p.d == 128) return attn_simt_launch<uint16_t, 128>(p, st);
    return attn_simt_launch<uint16_t, 64>(p, st);
  }
  if (p.d == 128) return attn_simt_launch<float, 128>(p, st);
  return attn_simt_launch<float, 64>(p, st);
}

int attn_simt_splits(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int n_sm) {
  const int g = Hq / Hkv;
  const int nq = kSRows / g;
  const long long tiles = (max_nodes + nq - 1) / nq;
  const long long base = static_cast<long long>(B) * Hkv * tiles;
  const long long target = 4LL * n_sm;   // two resident CTAs per SM, two waves
  long long s = (target + base - 1) / base;
  // splits of at least 64 keys (a short prefix over few tiles is split
  // finer: its CTAs are latency-bound, the combine costs one small kernel)
  const long long cap = std::max(1, (max_prefix + 63) / 64);
  s = std::min(s, cap);
  s = std::max(1LL, std::min(s, 64LL));
  return static_cast<int>(s);
}

}  // namespace tv
