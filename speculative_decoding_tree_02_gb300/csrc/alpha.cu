// tree_tv_alpha: alpha = sum_v min(p_v, q_v) = 1 - TV(p, q) per row, its
// running product along each branch, and the target's softmax mass of a given
// token (SpecOPD page §03: acceptance probability under exact rejection
// sampling is the distribution overlap; E2E-TV multiplies it along a branch.
// Graft page §3: coverage gain is target probability mass).
//
// bf16 rows whose length and stride are multiples of 8 (16 bytes): one read.
//   A cluster of 8 CTAs per row; CTA c copies its eighth of both rows into
//   shared memory with bulk copies and keeps it there.  Pass 1 on the slice:
//   max and sum of exp for p and q; the 8 partials are exchanged through
//   distributed shared memory, so every CTA knows the row's lse_p, lse_q.
//   Pass 2 on the same slice: sum of 2^(min(lp - Lp, lq - Lq) log2 e) (one
//   exponential per element, min taken on the exponents).  CTA 0 adds the 8
//   overlap partials.  Two CTAs per SM: one copies while the other computes.
// Other rows: two streaming passes over the logits:
//   pass A  grid (chunks, rows): chunk max and sum of exp for p and q
//   merge   warp per row: lse_p, lse_q (chunk order, deterministic)
//   pass B  grid (chunks, rows): sum of 2^(min(lp - Lp, lq - Lq) * log2 e)
//   final   warp per row: alpha, p_mass.
// Then one thread per branch: running product of alpha in row order.
#include <cuda_bf16.h>

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

// Workspace header: status word (nonzero: a copy wait ran out).
constexpr size_t kAlphaHdrBytes = 256;
__global__ void alpha_clear_kernel(int* err) {
  griddep_wait();
  griddep_release();
  *err = 0;
}

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
constexpr int kACluster = 8;
constexpr int kAClThreads = 256;
constexpr uint64_t kAlphaTimeoutNs = 2000000000ull;

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

// One row per cluster of 8 CTAs; S elements per CTA (multiple of 8).
__global__ void __cluster_dims__(kACluster, 1, 1) __launch_bounds__(kAClThreads, 2) alpha_cluster_kernel(
    const uint16_t* __restrict__ lp, const uint16_t* __restrict__ lq, int V, int64_t ld, int S,
    const int32_t* __restrict__ mass_tok, float* __restrict__ alpha, float* __restrict__ p_mass,
    int* __restrict__ err) {
  extern __shared__ __align__(128) uint8_t sm[];   // [S] p bf16, then [S] q bf16
  __shared__ __align__(8) uint64_t full;
  __shared__ float s_red[2][kAClThreads / 32];
  __shared__ float s_part[4];                        // this CTA's (mp, sp, mq, sq)
  __shared__ float s_ovl;                            // this CTA's overlap partial
  griddep_wait();
  griddep_release();
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int row = blockIdx.x / kACluster;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int base = static_cast<int>(rank) * S;
  const int n = max(0, min(S, V - base));            // elements of this slice (multiple of 8)
  const uint16_t* sp_ = reinterpret_cast<const uint16_t*>(sm);
  const uint16_t* sq_ = sp_ + S;
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a_smem(&full)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (n > 0) {
      const uint32_t bytes = static_cast<uint32_t>(n) * 2u;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a_smem(&full)), "r"(2u * bytes)
                   : "memory");
      const uint16_t* gp = lp + static_cast<int64_t>(row) * ld + base;
      const uint16_t* gq = lq + static_cast<int64_t>(row) * ld + base;
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       a_smem(sp_)),
                   "l"(gp), "r"(bytes), "r"(a_smem(&full))
                   : "memory");
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       a_smem(sq_)),
                   "l"(gq), "r"(bytes), "r"(a_smem(&full))
                   : "memory");
    } else {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a_smem(&full)) : "memory");
    }
  }
  __syncthreads();
  // bounded wait for the copies (every CTA still takes part in the cluster
  // barriers below, so a peer never waits on a CTA that gave up)
  bool ok = false;
  {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
      uint32_t done;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
          : "=r"(done)
          : "r"(a_smem(&full))
          : "memory");
      if (done) { ok = true; break; }
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (i == 0) t0 = t;
      else if (t - t0 > kAlphaTimeoutNs) break;
    }
  }
  if (!ok && tid == 0 && err) atomicExch(err, 1);
  const int nv = ok ? n : 0;                         // 8-element vectors below
  const uint4* vp = reinterpret_cast<const uint4*>(sp_);
  const uint4* vq = reinterpret_cast<const uint4*>(sq_);

  // pass 1: slice max and sum of exp for p and q
  __nv_bfloat162 pm2 = __float2bfloat162_rn(-INFINITY), qm2 = pm2;
  for (int i = tid; i < nv / 8; i += kAClThreads) {
    const uint4 a = vp[i], b = vq[i];
    pm2 = __hmax2(pm2, __hmax2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a.x),
                                       *reinterpret_cast<const __nv_bfloat162*>(&a.y)),
                               __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a.z),
                                       *reinterpret_cast<const __nv_bfloat162*>(&a.w))));
    qm2 = __hmax2(qm2, __hmax2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&b.x),
                                       *reinterpret_cast<const __nv_bfloat162*>(&b.y)),
                               __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&b.z),
                                       *reinterpret_cast<const __nv_bfloat162*>(&b.w))));
  }
  float mp = warp_max(fmaxf(__low2float(pm2), __high2float(pm2)));
  float mq = warp_max(fmaxf(__low2float(qm2), __high2float(qm2)));
  if (lane == 0) { s_red[0][warp] = mp; s_red[1][warp] = mq; }
  __syncthreads();
  mp = s_red[0][0];
  mq = s_red[1][0];
#pragma unroll
  for (int w = 1; w < kAClThreads / 32; ++w) { mp = fmaxf(mp, s_red[0][w]); mq = fmaxf(mq, s_red[1][w]); }
  __syncthreads();
  float sp = 0.f, sq = 0.f;
  if (mp != -INFINITY && mq != -INFINITY) {
    const float bp = mp * kLog2e, bq = mq * kLog2e;
    for (int i = tid; i < nv / 8; i += kAClThreads) {
      const uint4 a = vp[i], b = vq[i];
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sp += ex2(fmaf(bf16_lo(wa[k]), kLog2e, -bp)) + ex2(fmaf(bf16_hi(wa[k]), kLog2e, -bp));
        sq += ex2(fmaf(bf16_lo(wb[k]), kLog2e, -bq)) + ex2(fmaf(bf16_hi(wb[k]), kLog2e, -bq));
      }
    }
  }
  sp = warp_sum(sp);
  sq = warp_sum(sq);
  if (lane == 0) { s_red[0][warp] = sp; s_red[1][warp] = sq; }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int w = 0; w < kAClThreads / 32; ++w) { a += s_red[0][w]; b += s_red[1][w]; }
    s_part[0] = mp; s_part[1] = a; s_part[2] = mq; s_part[3] = b;
  }
  cluster_sync_all();   // every slice partial is visible to the whole cluster

  // row log-sum-exp (log2 units), the same in every CTA: slice order 0..7
  float Lp, Lq;
  {
    float m[kACluster][2], su[kACluster][2];
#pragma unroll
    for (int c = 0; c < kACluster; ++c) {
      m[c][0] = cluster_ld(&s_part[0], c);
      su[c][0] = cluster_ld(&s_part[1], c);
      m[c][1] = cluster_ld(&s_part[2], c);
      su[c][1] = cluster_ld(&s_part[3], c);
    }
    float Mp = -INFINITY, Mq = -INFINITY;
#pragma unroll
    for (int c = 0; c < kACluster; ++c) { Mp = fmaxf(Mp, m[c][0]); Mq = fmaxf(Mq, m[c][1]); }
    float Sp = 0.f, Sq = 0.f;
#pragma unroll
    for (int c = 0; c < kACluster; ++c) {
      if (m[c][0] != -INFINITY) Sp += su[c][0] * ex2((m[c][0] - Mp) * kLog2e);
      if (m[c][1] != -INFINITY) Sq += su[c][1] * ex2((m[c][1] - Mq) * kLog2e);
    }
    Lp = Mp * kLog2e + log2f(Sp);
    Lq = Mq * kLog2e + log2f(Sq);
  }

  // pass 2: overlap of the slice
  float ov = 0.f;
  for (int i = tid; i < nv / 8; i += kAClThreads) {
    const uint4 a = vp[i], b = vq[i];
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ov += ex2(fminf(fmaf(bf16_lo(wa[k]), kLog2e, -Lp), fmaf(bf16_lo(wb[k]), kLog2e, -Lq)));
      ov += ex2(fminf(fmaf(bf16_hi(wa[k]), kLog2e, -Lp), fmaf(bf16_hi(wb[k]), kLog2e, -Lq)));
    }
  }
  ov = warp_sum(ov);
  if (lane == 0) s_red[0][warp] = ov;
  __syncthreads();
  if (tid == 0) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kAClThreads / 32; ++w) a += s_red[0][w];
    s_ovl = a;
    if (mass_tok && p_mass) {
      const int t = mass_tok[row];
      if (t >= base && t < base + nv) p_mass[row] = ex2(fmaf(bf16_at(sp_ + (t - base)), kLog2e, -Lp));
      else if (rank == 0 && (t < 0 || t >= V)) p_mass[row] = 0.f;
    }
  }
  cluster_sync_all();
  if (rank == 0 && tid == 0) {
    float a = 0.f;
#pragma unroll
    for (int c = 0; c < kACluster; ++c) a += cluster_ld(&s_ovl, c);
    alpha[row] = a;
  }
  cluster_sync_all();   // no CTA leaves while CTA 0 still reads its shared memory
}

template <typename T>
int alpha_launch(const T* lp, const T* lq, int rows, int V, int64_t ld, const int32_t* branch_off,
                 int nb, const int32_t* mass_tok, float* alpha, float* alpha_prefix,
                 float* p_mass, void* ws, cudaStream_t st) {
  const int n_chunks = (V + kAChunk - 1) / kAChunk;
  const bool vec_ok =
      aligned(lp, 16) && aligned(lq, 16) && ((ld * static_cast<int64_t>(sizeof(T))) % 16 == 0);
  if constexpr (sizeof(T) == 2) {
    // one-read path: 16-byte rows and an eighth of a row that fits shared memory
    const int S = ((V + kACluster - 1) / kACluster + 7) / 8 * 8;
    const size_t smem = static_cast<size_t>(S) * 2 * sizeof(uint16_t);
    if (vec_ok && V % 8 == 0 && ld % 8 == 0 && smem <= 200 * 1024) {
      static int attr_bytes = 0;
      if (static_cast<int>(smem) > attr_bytes) {
        if (cudaFuncSetAttribute(alpha_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
          return TV_ECUDA;
        attr_bytes = static_cast<int>(smem);
      }
      int* err = static_cast<int*>(ws);
      int rc = launch_pdl(alpha_clear_kernel, dim3(1), dim3(1), 0, st, err);
      if (rc == TV_OK)
        rc = launch_pdl(alpha_cluster_kernel, dim3(rows * kACluster), dim3(kAClThreads), smem, st, lp, lq, V, ld, S,
                        mass_tok, alpha, p_mass, err);
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
