// tree_tv_alpha: alpha = sum_v min(p_v, q_v) = 1 - TV(p, q) per row, its
// running product along each branch, and the target's softmax mass of a given
// token (SpecOPD page §03: acceptance probability under exact rejection
// sampling is the distribution overlap; E2E-TV multiplies it along a branch.
// Graft page §3: coverage gain is target probability mass).
//
// bf16 rows whose length and stride are multiples of 8 (16 bytes): one read
// from HBM.  A cluster of 4 CTAs per row, CTA c on a quarter of both rows.
//   Pass 1 on the slice: running max and sum of exp for p and q; the 4
//   partials are exchanged through distributed shared memory, so every CTA
//   knows the row's lse_p, lse_q.  Pass 2 re-reads the slice, still in L2
//   (a quarter row per CTA keeps the reuse distance far below L2's size):
//   sum of 2^(min(lp - Lp, lq - Lq) log2 e), one exponential per element,
//   the min taken on the exponents.  CTA 0 adds the 4 overlap partials.
//   Clusters are persistent and step through rows.
// Other rows: two streaming passes over the logits:
//   pass A  grid (chunks, rows): chunk max and sum of exp for p and q
//   merge   warp per row: lse_p, lse_q (chunk order, deterministic)
//   pass B  grid (chunks, rows): sum of 2^(min(lp - Lp, lq - Lq) * log2 e)
//   final   warp per row: alpha, p_mass.
// Then one thread per branch: running product of alpha in row order.
#include <cuda_bf16.h>

#include <atomic>

#include "tv_common.cuh"

namespace tv {

constexpr int kAThreads = 256;
constexpr int kAPer = 16;                    // values per thread per input row
constexpr int kAChunk = kAThreads * kAPer;   // 4096 elements

struct AlphaLsePart { float mp, sp, mq, sq; };

__device__ __forceinline__ void aload8(const uint16_t* row, int e0, int V, bool vec_ok, float* o) {
  if (vec_ok && e0 + 8 <= V) {
    uint4 w = ldg_stream(row + e0);
    o[0] = bf16_lo(w.x); o[1] = bf16_hi(w.x); o[2] = bf16_lo(w.y); o[3] = bf16_hi(w.y);
    o[4] = bf16_lo(w.z); o[5] = bf16_hi(w.z); o[6] = bf16_lo(w.w); o[7] = bf16_hi(w.w);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = (e0 + q < V) ? bf16_at(row + e0 + q) : -INFINITY;
  }
}

__device__ __forceinline__ void aload8(const float* row, int e0, int V, bool vec_ok, float* o) {
  if (vec_ok && e0 + 8 <= V) {
    uint4 a = ldg_stream(row + e0);
    uint4 b = ldg_stream(row + e0 + 4);
    o[0] = __uint_as_float(a.x); o[1] = __uint_as_float(a.y);
    o[2] = __uint_as_float(a.z); o[3] = __uint_as_float(a.w);
    o[4] = __uint_as_float(b.x); o[5] = __uint_as_float(b.y);
    o[6] = __uint_as_float(b.z); o[7] = __uint_as_float(b.w);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = (e0 + q < V) ? row[e0 + q] : -INFINITY;
  }
}

template <typename T>
__device__ __forceinline__ void load_chunk(const T* row, int base, int V, bool vec_ok, float* v) {
#pragma unroll
  for (int j = 0; j < kAPer / 8; ++j)
    aload8(row, base + (j * kAThreads + threadIdx.x) * 8, V, vec_ok, v + 8 * j);
}

__device__ __forceinline__ float block_sum(float v, float* s_red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kAThreads / 32; ++w) t += s_red[w];
  return t;
}

__device__ __forceinline__ float block_max(float v, float* s_red) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = s_red[0];
#pragma unroll
  for (int w = 1; w < kAThreads / 32; ++w) t = fmaxf(t, s_red[w]);
  return t;
}

template <typename T>
__global__ void __launch_bounds__(kAThreads) alpha_lse_kernel(
    const T* __restrict__ lp, const T* __restrict__ lq, int V, int64_t ld, bool vec_ok,
    AlphaLsePart* __restrict__ part) {
  __shared__ float s_red[kAThreads / 32];
  const int row = blockIdx.y, chunk = blockIdx.x, base = chunk * kAChunk;
  float vp[kAPer], vq[kAPer];
  load_chunk(lp + static_cast<int64_t>(row) * ld, base, V, vec_ok, vp);
  load_chunk(lq + static_cast<int64_t>(row) * ld, base, V, vec_ok, vq);
  float mp = vp[0], mq = vq[0];
#pragma unroll
  for (int t = 1; t < kAPer; ++t) { mp = fmaxf(mp, vp[t]); mq = fmaxf(mq, vq[t]); }
  mp = block_max(mp, s_red);
  mq = block_max(mq, s_red);
  float sp = 0.f, sq = 0.f;
  const float bp = mp * kLog2e, bq = mq * kLog2e;
#pragma unroll
  for (int t = 0; t < kAPer; ++t) {
    sp += ex2(fmaf(vp[t], kLog2e, -bp));
    sq += ex2(fmaf(vq[t], kLog2e, -bq));
  }
  sp = block_sum(sp, s_red);
  sq = block_sum(sq, s_red);
  if (threadIdx.x == 0)
    part[static_cast<int64_t>(row) * gridDim.x + chunk] = AlphaLsePart{mp, sp, mq, sq};
}

// lse2[row] = (Lp, Lq) in log2 units of the logits: L = M*log2e + log2(S).
__global__ void __launch_bounds__(128) alpha_lse_merge_kernel(
    const AlphaLsePart* __restrict__ part, int n_chunks, int rows, float2* __restrict__ lse2) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const AlphaLsePart* p = part + static_cast<int64_t>(row) * n_chunks;
  float Mp = -INFINITY, Mq = -INFINITY;
  for (int c = lane; c < n_chunks; c += 32) { Mp = fmaxf(Mp, p[c].mp); Mq = fmaxf(Mq, p[c].mq); }
  Mp = warp_max(Mp);
  Mq = warp_max(Mq);
  float Sp = 0.f, Sq = 0.f;
  for (int c = lane; c < n_chunks; c += 32) {
    Sp += p[c].sp * ex2((p[c].mp - Mp) * kLog2e);
    Sq += p[c].sq * ex2((p[c].mq - Mq) * kLog2e);
  }
  Sp = warp_sum(Sp);
  Sq = warp_sum(Sq);
  if (lane == 0) lse2[row] = make_float2(Mp * kLog2e + log2f(Sp), Mq * kLog2e + log2f(Sq));
}

template <typename T>
__global__ void __launch_bounds__(kAThreads) alpha_overlap_kernel(
    const T* __restrict__ lp, const T* __restrict__ lq, int V, int64_t ld, bool vec_ok,
    const float2* __restrict__ lse2, float* __restrict__ part) {
  __shared__ float s_red[kAThreads / 32];
  const int row = blockIdx.y, chunk = blockIdx.x, base = chunk * kAChunk;
  float vp[kAPer], vq[kAPer];
  load_chunk(lp + static_cast<int64_t>(row) * ld, base, V, vec_ok, vp);
  load_chunk(lq + static_cast<int64_t>(row) * ld, base, V, vec_ok, vq);
  const float2 L = lse2[row];
  float a = 0.f;
#pragma unroll
  for (int t = 0; t < kAPer; ++t)
    a += ex2(fminf(fmaf(vp[t], kLog2e, -L.x), fmaf(vq[t], kLog2e, -L.y)));
  a = block_sum(a, s_red);
  if (threadIdx.x == 0) part[static_cast<int64_t>(row) * gridDim.x + chunk] = a;
}

template <typename T>
__global__ void __launch_bounds__(128) alpha_final_kernel(
    const float* __restrict__ part, int n_chunks, int rows, const T* __restrict__ lp, int V,
    int64_t ld, const float2* __restrict__ lse2, const int32_t* __restrict__ mass_tok,
    float* __restrict__ alpha, float* __restrict__ p_mass) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  float a = 0.f;
  for (int c = lane; c < n_chunks; c += 32) a += part[static_cast<int64_t>(row) * n_chunks + c];
  a = warp_sum(a);
  if (lane == 0) {
    alpha[row] = a;
    if (mass_tok && p_mass) {
      const int t = mass_tok[row];
      float m = 0.f;
      if (t >= 0 && t < V) {
        const T* x = lp + static_cast<int64_t>(row) * ld + t;
        float xv;
        if constexpr (sizeof(T) == 2) xv = bf16_at(reinterpret_cast<const uint16_t*>(x));
        else xv = *reinterpret_cast<const float*>(x);
        m = ex2(fmaf(xv, kLog2e, -lse2[row].x));
      }
      p_mass[row] = m;
    }
  }
}

// Workspace: a reserved 256-byte header, then the two-pass partials.
constexpr size_t kAlphaHdrBytes = 256;

__global__ void alpha_prefix_kernel(const float* __restrict__ alpha, int rows,
                                    const int32_t* __restrict__ branch_off, int nb,
                                    float* __restrict__ prefix) {
  griddep_wait();
  griddep_release();
  // rows outside every branch keep 1
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x)
    prefix[r] = 1.f;
  __syncthreads();
  if (blockIdx.x != 0) return;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    int r0 = max(branch_off[b], 0), r1 = min(branch_off[b + 1], rows);
    float run = 1.f;
    for (int r = r0; r < r1; ++r) {
      run *= alpha[r];
      prefix[r] = run;
    }
  }
}

// ------------------------------------------------------------ one-read path
constexpr int kACluster = 4;
constexpr int kAClThreads = 512;

__device__ __forceinline__ uint32_t a_smem(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// float at the same shared-memory offset in CTA `rank` of this cluster
__device__ __forceinline__ float cluster_ld(const float* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a_smem(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ float bmax8(uint4 x) {
  const __nv_bfloat162 h = __hmax2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&x.x),
                                           *reinterpret_cast<const __nv_bfloat162*>(&x.y)),
                                   __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&x.z),
                                           *reinterpret_cast<const __nv_bfloat162*>(&x.w)));
  return fmaxf(__low2float(h), __high2float(h));
}
// Packed fp32 pairs (sm_100 family): one FMA or add instruction computes two
// values, each rounded as the scalar instruction would round it, so the two
// passes issue about a fifth fewer instructions per element.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void upk2(uint64_t d, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the two bf16 of word w as an fp32 pair (low half first)
__device__ __forceinline__ uint64_t bpair(uint32_t w) { return pk2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ uint64_t ex2_pair(uint64_t a) {
  float lo, hi;
  upk2(a, lo, hi);
  return pk2(ex2(lo), ex2(hi));
}
// running (max, pair of partial sums) of exp over 8 bf16 logits
__device__ __forceinline__ void online8(uint4 x, float& m, uint64_t& s) {
  const float m8 = bmax8(x);
  if (m8 > m) {   // rescale (the sums are 0 while m is -inf)
    const float f = ex2((m - m8) * kLog2e);
    float a, b;
    upk2(s, a, b);
    s = pk2(a * f, b * f);
    m = m8;
  }
  if (m != -INFINITY) {
    const float bm = m * kLog2e;
    const uint64_t l2 = pk2(kLog2e, kLog2e), nb = pk2(-bm, -bm);
    s = add2(s, ex2_pair(fma2(bpair(x.x), l2, nb)));
    s = add2(s, ex2_pair(fma2(bpair(x.y), l2, nb)));
    s = add2(s, ex2_pair(fma2(bpair(x.z), l2, nb)));
    s = add2(s, ex2_pair(fma2(bpair(x.w), l2, nb)));
  }
}
__device__ __forceinline__ void online8(uint4 x, float& m, float& s0, float& s1) {
  uint64_t s = pk2(s0, s1);
  online8(x, m, s);
  upk2(s, s0, s1);
}
// sum over 8 elements of 2^min(lp log2e - Lp, lq log2e - Lq)
__device__ __forceinline__ void overlap8(uint4 x, uint4 y, float Lp, float Lq, float& a, float& b) {
  const uint64_t l2 = pk2(kLog2e, kLog2e), np = pk2(-Lp, -Lp), nq = pk2(-Lq, -Lq);
  uint64_t acc = pk2(a, b);
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float p0, p1, q0, q1;
    upk2(fma2(bpair(xs[c]), l2, np), p0, p1);
    upk2(fma2(bpair(ys[c]), l2, nq), q0, q1);
    acc = add2(acc, pk2(ex2(fminf(p0, q0)), ex2(fminf(p1, q1))));
  }
  upk2(acc, a, b);
}
// Persistent clusters of 4 CTAs; cluster c takes rows c, c + NC, ...; CTA r
// of a cluster owns elements [r S, (r + 1) S) of each row (S a multiple of 8).
// Per row: pass 1 reads the slice from HBM (running max and sum of exp), one
// cluster barrier makes the 4 slice partials of this row and the 4 overlap
// partials of the previous row visible, warp 0 forms the row's lse, pass 2
// re-reads the slice, which a quarter row ago was read into L2, and sums the
// overlap.  CTA 0 adds the previous row's overlap partials.
__global__ void __cluster_dims__(kACluster, 1, 1) __launch_bounds__(kAClThreads, 2) alpha_cluster_kernel(
    const uint16_t* __restrict__ lp, const uint16_t* __restrict__ lq, int rows, int V, int64_t ld, int S,
    const int32_t* __restrict__ mass_tok, float* __restrict__ alpha, float* __restrict__ p_mass) {
  __shared__ float s_red[4][kAClThreads / 32];
  __shared__ float s_ov[kAClThreads / 32];
  __shared__ float s_part[2][4];   // (mp, sp, mq, sq) of the rows in flight, by parity
  __shared__ float s_ovl[2];       // overlap partials, by parity
  __shared__ float s_L[2];         // the current row's lse of p and q (log2 units)
  griddep_wait();
  griddep_release();
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int NC = gridDim.x / kACluster, cl = blockIdx.x / kACluster;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int base = static_cast<int>(rank) * S;
  const int n8 = max(0, min(S, V - base)) / 8;   // 16-byte words of this slice
  const int K = cl < rows ? (rows - cl + NC - 1) / NC : 0;
  for (int k = 0; k < K; ++k) {
    const int b = k & 1, row = cl + k * NC;
    const uint4* gp = reinterpret_cast<const uint4*>(lp + static_cast<int64_t>(row) * ld + base);
    const uint4* gq = reinterpret_cast<const uint4*>(lq + static_cast<int64_t>(row) * ld + base);
    // pass 1
    float mp = -INFINITY, mq = -INFINITY, sp0 = 0.f, sp1 = 0.f, sq0 = 0.f, sq1 = 0.f;
    int i = tid;
    for (; i + 2 * kAClThreads < n8; i += 3 * kAClThreads) {   // three vector pairs in flight
      const uint4 x0 = __ldg(gp + i), y0 = __ldg(gq + i);
      const uint4 x1 = __ldg(gp + i + kAClThreads), y1 = __ldg(gq + i + kAClThreads);
      const uint4 x2 = __ldg(gp + i + 2 * kAClThreads), y2 = __ldg(gq + i + 2 * kAClThreads);
      online8(x0, mp, sp0, sp1);
      online8(y0, mq, sq0, sq1);
      online8(x1, mp, sp0, sp1);
      online8(y1, mq, sq0, sq1);
      online8(x2, mp, sp0, sp1);
      online8(y2, mq, sq0, sq1);
    }
    for (; i < n8; i += kAClThreads) {
      online8(__ldg(gp + i), mp, sp0, sp1);
      online8(__ldg(gq + i), mq, sq0, sq1);
    }
    float spp = sp0 + sp1, sqq = sq0 + sq1;
    {
      const float Mp = warp_max(mp), Mq = warp_max(mq);
      spp = warp_sum(mp == -INFINITY ? 0.f : spp * ex2((mp - Mp) * kLog2e));
      sqq = warp_sum(mq == -INFINITY ? 0.f : sqq * ex2((mq - Mq) * kLog2e));
      mp = Mp;
      mq = Mq;
    }
    if (lane == 0) { s_red[0][warp] = mp; s_red[1][warp] = spp; s_red[2][warp] = mq; s_red[3][warp] = sqq; }
    __syncthreads();
    if (warp == 0) {   // CTA partial: lane w holds warp w's pair
      constexpr int W = kAClThreads / 32;
      const float m0 = lane < W ? s_red[0][lane] : -INFINITY, s0 = lane < W ? s_red[1][lane] : 0.f;
      const float m1 = lane < W ? s_red[2][lane] : -INFINITY, s1 = lane < W ? s_red[3][lane] : 0.f;
      const float Mp = warp_max(m0), Mq = warp_max(m1);
      const float x = warp_sum(m0 == -INFINITY ? 0.f : s0 * ex2((m0 - Mp) * kLog2e));
      const float y = warp_sum(m1 == -INFINITY ? 0.f : s1 * ex2((m1 - Mq) * kLog2e));
      if (lane == 0) { s_part[b][0] = Mp; s_part[b][1] = x; s_part[b][2] = Mq; s_part[b][3] = y; }
    }
    cluster_sync_all();   // this row's slice partials and the previous row's overlaps are visible
    if (warp == 0) {
      if (rank == 0 && k > 0) {
        const float o = lane < kACluster ? cluster_ld(&s_ovl[b ^ 1], lane) : 0.f;
        float x = 0.f;
#pragma unroll
        for (int c = 0; c < kACluster; ++c) x += __shfl_sync(0xffffffffu, o, c);
        if (lane == 0) alpha[row - NC] = x;
      }
      float m0 = -INFINITY, s0 = 0.f, m1 = -INFINITY, s1 = 0.f;
      if (lane < kACluster) {
        m0 = cluster_ld(&s_part[b][0], lane);
        s0 = cluster_ld(&s_part[b][1], lane);
        m1 = cluster_ld(&s_part[b][2], lane);
        s1 = cluster_ld(&s_part[b][3], lane);
      }
      const float Mp = warp_max(m0), Mq = warp_max(m1);
      const float tp = m0 == -INFINITY ? 0.f : s0 * ex2((m0 - Mp) * kLog2e);
      const float tq = m1 == -INFINITY ? 0.f : s1 * ex2((m1 - Mq) * kLog2e);
      float Sp = 0.f, Sq = 0.f;   // slice order
#pragma unroll
      for (int c = 0; c < kACluster; ++c) {
        Sp += __shfl_sync(0xffffffffu, tp, c);
        Sq += __shfl_sync(0xffffffffu, tq, c);
      }
      if (lane == 0) {
        s_L[0] = Mp * kLog2e + log2f(Sp);
        s_L[1] = Mq * kLog2e + log2f(Sq);
      }
    }
    __syncthreads();
    const float Lp = s_L[0], Lq = s_L[1];
    // pass 2
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    i = tid;
    for (; i + 2 * kAClThreads < n8; i += 3 * kAClThreads) {
      const uint4 x0 = __ldg(gp + i), y0 = __ldg(gq + i);
      const uint4 x1 = __ldg(gp + i + kAClThreads), y1 = __ldg(gq + i + kAClThreads);
      const uint4 x2 = __ldg(gp + i + 2 * kAClThreads), y2 = __ldg(gq + i + 2 * kAClThreads);
      overlap8(x0, y0, Lp, Lq, o0, o1);
      overlap8(x1, y1, Lp, Lq, o2, o3);
      overlap8(x2, y2, Lp, Lq, o0, o3);
    }
    for (; i < n8; i += kAClThreads) overlap8(__ldg(gp + i), __ldg(gq + i), Lp, Lq, o0, o1);
    const float ov = warp_sum((o0 + o1) + (o2 + o3));
    if (lane == 0) s_ov[warp] = ov;
    __syncthreads();
    if (warp == 0) {
      const float x = warp_sum(lane < kAClThreads / 32 ? s_ov[lane] : 0.f);
      if (lane == 0) {
        s_ovl[b] = x;
        if (mass_tok && p_mass) {
          const int t = mass_tok[row];
          if (t >= base && t < base + 8 * n8)
            p_mass[row] = ex2(fmaf(bf16_at(lp + static_cast<int64_t>(row) * ld + t), kLog2e, -Lp));
          else if (rank == 0 && (t < 0 || t >= V))
            p_mass[row] = 0.f;
        }
      }
    }
  }
  cluster_sync_all();   // the last row's overlap partials
  if (rank == 0 && warp == 0 && K > 0) {
    const float o = lane < kACluster ? cluster_ld(&s_ovl[(K - 1) & 1], lane) : 0.f;
    float x = 0.f;
#pragma unroll
    for (int c = 0; c < kACluster; ++c) x += __shfl_sync(0xffffffffu, o, c);
    if (lane == 0) alpha[cl + (K - 1) * NC] = x;
  }
  cluster_sync_all();   // no CTA leaves while CTA 0 still reads its shared memory
}

// Clusters that fit at once (a cluster sits in one GPC, so this can be below
// the SM count times CTAs per SM over the cluster size).
static int alpha_resident_clusters() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];   // per device; 0: not measured yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  if (const int c = cache[dev].load(std::memory_order_relaxed)) return c;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kACluster);
  cfg.blockDim = dim3(kAClThreads);
  cfg.dynamicSmemBytes = 0;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, alpha_cluster_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = std::max(1, 2 * sm_count() / kACluster);
  }
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <typename T>
int alpha_launch(const T* lp, const T* lq, int rows, int V, int64_t ld, const int32_t* branch_off,
                 int nb, const int32_t* mass_tok, float* alpha, float* alpha_prefix,
                 float* p_mass, void* ws, cudaStream_t st) {
  const int n_chunks = (V + kAChunk - 1) / kAChunk;
  const bool vec_ok =
      aligned(lp, 16) && aligned(lq, 16) && ((ld * static_cast<int64_t>(sizeof(T))) % 16 == 0);
  if constexpr (sizeof(T) == 2) {
    // one-read path: 16-byte rows
    if (vec_ok && V % 8 == 0 && ld % 8 == 0) {
      const int S = ((V + kACluster - 1) / kACluster + 7) / 8 * 8;
      const int NC = std::max(1, std::min(rows, alpha_resident_clusters()));
      int rc = launch_pdl(alpha_cluster_kernel, dim3(NC * kACluster), dim3(kAClThreads), 0, st, lp, lq, rows, V, ld,
                          S, mass_tok, alpha, p_mass);
      if (rc == TV_OK && alpha_prefix && branch_off)
        rc = launch_pdl(alpha_prefix_kernel, dim3(1), dim3(256), 0, st, alpha, rows, branch_off, nb, alpha_prefix);
      return rc;
    }
  }
  char* w = static_cast<char*>(ws) + kAlphaHdrBytes;
  auto* lpart = reinterpret_cast<AlphaLsePart*>(w);
  w += static_cast<size_t>(rows) * n_chunks * sizeof(AlphaLsePart);
  auto* lse2 = reinterpret_cast<float2*>(w);
  w += static_cast<size_t>(rows) * sizeof(float2);
  auto* apart = reinterpret_cast<float*>(w);
  dim3 g(n_chunks, rows);
  alpha_lse_kernel<T><<<g, kAThreads, 0, st>>>(lp, lq, V, ld, vec_ok, lpart);
  alpha_lse_merge_kernel<<<(rows + 3) / 4, 128, 0, st>>>(lpart, n_chunks, rows, lse2);
  alpha_overlap_kernel<T><<<g, kAThreads, 0, st>>>(lp, lq, V, ld, vec_ok, lse2, apart);
  alpha_final_kernel<T><<<(rows + 3) / 4, 128, 0, st>>>(apart, n_chunks, rows, lp, V, ld, lse2,
                                                         mass_tok, alpha, p_mass);
  if (alpha_prefix && branch_off) {
    // single CTA: the "1" fill and the branch products are ordered by __syncthreads
    alpha_prefix_kernel<<<1, 256, 0, st>>>(alpha, rows, branch_off, nb, alpha_prefix);
  }
  return launch_status();
}

}  // namespace tv

TV_API size_t tree_tv_alpha_workspace_size(int rows, int V) {
  if (rows <= 0 || V <= 0) return 0;
  const size_t n_chunks = (static_cast<size_t>(V) + tv::kAChunk - 1) / tv::kAChunk;
  return tv::kAlphaHdrBytes + static_cast<size_t>(rows) *
         (n_chunks * sizeof(tv::AlphaLsePart) + sizeof(float2) + n_chunks * sizeof(float));
}

TV_API int tree_tv_alpha(const void* p_logits, const void* q_logits, int dtype, int rows, int V,
                         int64_t ld, const int32_t* branch_off, int nb, const int32_t* mass_tok,
                         float* alpha, float* alpha_prefix, float* p_mass, void* ws,
                         size_t ws_bytes, tv_stream_t stream) {
  if (rows < 0 || V <= 0 || ld < V || nb < 0) return TV_EINVAL;
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_EINVAL;
  if (rows == 0) return TV_OK;
  if (!p_logits || !q_logits || !alpha) return TV_EINVAL;
  if (alpha_prefix && !branch_off) return TV_EINVAL;
  if (p_mass && !mass_tok) return TV_EINVAL;
  if (rows > 65535) return TV_EUNSUPPORTED;
  const size_t need = tree_tv_alpha_workspace_size(rows, V);
  if (!ws || ws_bytes < need || !tv::aligned(ws, 16)) return TV_EWORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TV_BF16)
    return tv::alpha_launch(static_cast<const uint16_t*>(p_logits),
                            static_cast<const uint16_t*>(q_logits), rows, V, ld, branch_off, nb,
                            mass_tok, alpha, alpha_prefix, p_mass, ws, st);
  return tv::alpha_launch(static_cast<const float*>(p_logits), static_cast<const float*>(q_logits),
                          rows, V, ld, branch_off, nb, mass_tok, alpha, alpha_prefix, p_mass, ws,
                          st);
}
