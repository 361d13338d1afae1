// dcut_select: D-cut prefix-product scores and batch-global budget selection
// (D-cut page, technical summary §2 core mechanism and pipeline; §1 B x (D+1)).
//
// One CTA of 1024 threads (T = B(D+1) <= 8192):
//   1. one thread per request forms s[r,j] = s[r,j-1] * conf[r,j-1] strictly
//      left to right in fp32 (products only, so nothing can be contracted);
//   2. the positions are sorted by the 64-bit key (~bits(s), t): scores are
//      non-negative, so their IEEE bits order like the values, and the key
//      order is (s desc, position asc) = (s desc, r asc, j asc).  A bitonic
//      network over n = 1024 E keys (E per thread, padding keys sort last):
//      compare distances below E stay in a thread, distances below 32 E are
//      warp shuffles, only the larger ones go through shared memory (15 of
//      the 55 stages for T <= 1024, one barrier each);
//   3. rank(t) = sorted position; t is kept for budget K iff rank(t) < K;
//   4. one block-wide exclusive scan of the keep counts of every budget at
//      once (two budgets per 32-bit word) gives the packed slot of every kept
//      position and the per-request offsets; one warp per request counts the
//      lengths (no assumption that the kept set is a prefix).
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "tv_common.cuh"

namespace tv {

constexpr int kDcutMaxPos = 8192;
constexpr int kDcutMaxRho = 8;
constexpr int kDcutThreads = 1024;

struct DcutK { int K[kDcutMaxRho]; };

// Exclusive scan of four words per thread across the 1024-thread block, each
// word holding two 16-bit counts (totals stay below 2^16: T <= 8192).
__device__ __forceinline__ uint4 block_excl_scan4(uint4 x, uint4* s_w, uint4* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint4 v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint4 y;
    y.x = __shfl_up_sync(0xffffffffu, v.x, o);
    y.y = __shfl_up_sync(0xffffffffu, v.y, o);
    y.z = __shfl_up_sync(0xffffffffu, v.z, o);
    y.w = __shfl_up_sync(0xffffffffu, v.w, o);
    if (lane >= o) { v.x += y.x; v.y += y.y; v.z += y.z; v.w += y.w; }
  }
  if (lane == 31) s_w[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const uint4 w = s_w[lane];
    uint4 iw = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint4 y;
      y.x = __shfl_up_sync(0xffffffffu, iw.x, o);
      y.y = __shfl_up_sync(0xffffffffu, iw.y, o);
      y.z = __shfl_up_sync(0xffffffffu, iw.z, o);
      y.w = __shfl_up_sync(0xffffffffu, iw.w, o);
      if (lane >= o) { iw.x += y.x; iw.y += y.y; iw.z += y.z; iw.w += y.w; }
    }
    s_w[lane] = make_uint4(iw.x - w.x, iw.y - w.y, iw.z - w.z, iw.w - w.w);   // exclusive
    if (lane == 31) s_w[32] = iw;                                              // block total
  }
  __syncthreads();
  const uint4 base = s_w[warp];
  *total = s_w[32];
  return make_uint4(base.x + v.x - x.x, base.y + v.y - x.y, base.z + v.z - x.z, base.w + v.w - x.w);
}

__device__ __forceinline__ int half16(const uint4& w, int a) {
  const uint32_t word = (a >> 1) == 0 ? w.x : (a >> 1) == 1 ? w.y : (a >> 1) == 2 ? w.z : w.w;
  return static_cast<int>((a & 1) ? (word >> 16) : (word & 0xffffu));
}

// E keys per thread; element i = tid * E + e of the n = 1024 E sorted keys.
template <int E>
__global__ void __launch_bounds__(kDcutThreads, 1) dcut_kernel(
    const float* __restrict__ conf, int B, int D, int n_rho, DcutK ks, float* __restrict__ score,
    uint8_t* __restrict__ keep, int32_t* __restrict__ keep_len, int32_t* __restrict__ pack_off,
    int32_t* __restrict__ pack_idx) {
  constexpr int n = kDcutThreads * E;
  extern __shared__ unsigned long long s_key[];                       // [n] sort keys
  int* s_rank = reinterpret_cast<int*>(s_key + kDcutMaxPos);          // [T]
  __shared__ uint4 s_w[33];
  griddep_wait();
  griddep_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = D + 1;
  const int T = B * N;

  // 1. confidences into shared memory with one coalesced pass (they sit in
  //    the rank array's space, which is not needed until step 3)
  float* s_conf = reinterpret_cast<float*>(s_rank);
  for (int i = tid; i < B * D; i += kDcutThreads) s_conf[i] = conf[i];
  __syncthreads();
  for (int r = tid; r < B; r += kDcutThreads) {
    float s = 1.f;
    for (int j = 0; j <= D; ++j) {
      if (j > 0) s = __fmul_rn(s, s_conf[r * D + j - 1]);
      const int t = r * N + j;
      s_key[t] = (static_cast<unsigned long long>(~__float_as_uint(s)) << 32) | static_cast<unsigned>(t);
    }
  }
  for (int t = T + tid; t < n; t += kDcutThreads) s_key[t] = ~0ull;
  __syncthreads();
  // scores out, coalesced (the key's high word holds the score's bits)
  for (int t = tid; t < T; t += kDcutThreads) score[t] = __uint_as_float(~static_cast<unsigned>(s_key[t] >> 32));
  unsigned long long key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) key[e] = s_key[tid * E + e];
  __syncthreads();   // keys read before the network writes them back

  // 2. bitonic network, ascending keys
  for (int k = 2; k <= n; k <<= 1) {
    int j = k >> 1;
    if (j >= 32 * E) {   // cross-warp distances through shared memory
#pragma unroll
      for (int e = 0; e < E; ++e) s_key[tid * E + e] = key[e];
      __syncthreads();
      for (; j >= 32 * E; j >>= 1) {
#pragma unroll
        for (int q = 0; q < E; ++q) {
          const int i = q * kDcutThreads + tid;
          const int p = i ^ j;
          if (p > i) {
            const unsigned long long a = s_key[i], b = s_key[p];
            if ((a > b) == ((i & k) == 0)) { s_key[i] = b; s_key[p] = a; }
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int e = 0; e < E; ++e) key[e] = s_key[tid * E + e];
    }
    for (; j >= E; j >>= 1) {   // partner in lane ^ (j / E), same slot
      const int m = j / E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, key[e], m);
        const int i = tid * E + e;
        const bool take_min = ((i & j) == 0) == ((i & k) == 0);
        key[e] = take_min ? (o < key[e] ? o : key[e]) : (o > key[e] ? o : key[e]);
      }
    }
#pragma unroll
    for (int jj = E >> 1; jj >= 1; jj >>= 1) {   // partner in the same thread
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if ((e & jj) == 0) {
          const int i = tid * E + e;
          const unsigned long long a = key[e], b = key[e | jj];
          if ((a > b) == ((i & k) == 0)) { key[e] = b; key[e | jj] = a; }
        }
      }
    }
  }
  // 3. rank of each position (padding keys carry t = 0xffffffff)
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const unsigned t = static_cast<unsigned>(key[e] & 0xffffffffu);
    if (t < static_cast<unsigned>(T)) s_rank[t] = tid * E + e;
  }
  __syncthreads();

  // 4. flags and counts of every budget, one scan for all of them
  const int per = (T + kDcutThreads - 1) / kDcutThreads;   // consecutive positions per thread (<= E)
  const int t0 = tid * per;
  int rk[E];
  uint32_t cw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int q = 0; q < E; ++q) {
    const int t = t0 + q;
    rk[q] = (q < per && t < T) ? s_rank[t] : INT32_MAX;
#pragma unroll
    for (int a = 0; a < kDcutMaxRho; ++a)
      if (a < n_rho && rk[q] < ks.K[a]) cw[a >> 1] += (a & 1) ? 0x10000u : 1u;
  }
  uint4 total;
  const uint4 ex = block_excl_scan4(make_uint4(cw[0], cw[1], cw[2], cw[3]), s_w, &total);
#pragma unroll
  for (int a = 0; a < kDcutMaxRho; ++a) {
    if (a >= n_rho) break;
    const int K = ks.K[a];
    const int tot = half16(total, a);
    int o = half16(ex, a);
    uint8_t* kp = keep + static_cast<int64_t>(a) * T;
    int32_t* pi = pack_idx ? pack_idx + static_cast<int64_t>(a) * T : nullptr;
#pragma unroll
    for (int q = 0; q < E; ++q) {
      const int t = t0 + q;
      if (q < per && t < T) {
        const int f = rk[q] < K;
        kp[t] = static_cast<uint8_t>(f);
        const int r = t / N;
        if (t == r * N && pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + r] = o;   // kept before request r
        if (f && pi) pi[o] = t;
        o += f;
      }
    }
    if (tid == 0 && pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + B] = tot;
    if (pi)
      for (int q = tot + tid; q < T; q += kDcutThreads) pi[q] = -1;
  }
  // keep_len[r]: one warp per request, lanes over its positions
  for (int r = warp; r < B; r += kDcutThreads / 32) {
    int c[kDcutMaxRho] = {};
    for (int j = lane; j < N; j += 32) {
      const int x = s_rank[r * N + j];
#pragma unroll
      for (int a = 0; a < kDcutMaxRho; ++a) c[a] += a < n_rho && x < ks.K[a];
    }
#pragma unroll
    for (int a = 0; a < kDcutMaxRho; ++a) {
      if (a < n_rho) {
        const int sum = __reduce_add_sync(0xffffffffu, c[a]);
        if (lane == 0) keep_len[static_cast<int64_t>(a) * B + r] = sum;
      }
    }
  }
}

// Cluster form for T <= 2048 (the single-CTA network above is latency-bound:
// ~11k SM cycles for its 55 stages at T = 1024).  A cluster of 8 CTAs; every
// CTA forms all T keys (same left-to-right products), then CTA c ranks its
// eighth of the positions by counting, over all T keys, those that order
// before it (rank = #{u : key_u < key_t}; keys are distinct).  Position t is
// kept for budget K iff rank(t) < K, so each CTA knows the flags of its own
// positions at once; it stores its kept counts into every CTA's shared memory,
// and after one cluster barrier the counts of the CTAs before it give the
// packed slot of its first kept position.  It writes the outputs of its
// positions and the lengths of the requests that start in its range (reading
// the ranks of a request's later positions from the CTAs that hold them).
constexpr int kDcCl = 8;
constexpr int kDcClMaxT = 2048;

__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return remote;
}
__device__ __forceinline__ void st_cluster_s32(int* p, uint32_t rank, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(cluster_addr(p, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_cluster_s32(const int* p, uint32_t rank) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}

__global__ void __cluster_dims__(kDcCl, 1, 1) __launch_bounds__(kDcutThreads, 1) dcut_cluster_kernel(
    const float* __restrict__ conf, int B, int D, int n_rho, DcutK ks, float* __restrict__ score,
    uint8_t* __restrict__ keep, int32_t* __restrict__ keep_len, int32_t* __restrict__ pack_off,
    int32_t* __restrict__ pack_idx) {
  __shared__ __align__(16) unsigned long long s_key[kDcClMaxT + 4];
  __shared__ __align__(16) uint32_t s_hi[kDcClMaxT + 4];   // score words of the keys
  __shared__ float s_conf[kDcClMaxT];
  __shared__ int s_part[2 * kDcutThreads];
  __shared__ int s_rank[kDcClMaxT / kDcCl];                // ranks of this CTA's positions
  __shared__ int s_wcnt[kDcClMaxT / kDcCl / 32][kDcutMaxRho];   // kept per warp of the range
  __shared__ int s_ccnt[kDcCl][kDcutMaxRho];               // kept per CTA (written by each CTA)
  uint32_t crank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  // this CTA has started; the matching wait comes before the first remote store
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  griddep_wait();
  griddep_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = D + 1;
  const int T = B * N;
  const int P = (T + kDcCl - 1) / kDcCl;   // positions per CTA (<= 256)
  const int p0 = min(T, static_cast<int>(crank) * P), p1 = min(T, p0 + P);

  // 1. keys of every position: s[r,j] = ((1 * c[r,0]) * c[r,1]) ... * c[r,j-1] in fp32
  for (int i = tid; i < B * D; i += kDcutThreads) s_conf[i] = conf[i];
  __syncthreads();
  for (int t = tid; t < T; t += kDcutThreads) {
    const int r = t / N, j = t - r * N;
    const float* c = s_conf + r * D;
    float sc = 1.f;
    for (int i = 0; i < j; ++i) sc = __fmul_rn(sc, c[i]);
    s_key[t] = (static_cast<unsigned long long>(~__float_as_uint(sc)) << 32) | static_cast<unsigned>(t);
    s_hi[t] = ~__float_as_uint(sc);
  }
  if (tid < 4) {   // padding: orders after every key
    s_key[T + tid] = ~0ull;
    s_hi[T + tid] = ~0u;
  }
  __syncthreads();

  // 2. ranks of this CTA's positions.  Warp = (key sub-range, group of 64
  //    positions x0 .. x0 + 63); lane l ranks x0 + l and x0 + 32 + l.
  //    key_u < key_x compares the score words and breaks ties by position,
  //    so keys below x0 need hi_u <= hi_x, keys at or above x0 + 64 need
  //    hi_u < hi_x, and only the four-key groups that meet the warp's own
  //    positions take the full 64-bit compare.
  const int G = P <= 64 ? 1 : P <= 128 ? 2 : 4;
  const int SR = 32 / G;
  {
    const int g = warp % G, sr = warp / G;
    const int x0 = p0 + g * 64, xa = x0 + lane, xb = xa + 32;
    const unsigned long long ka = xa < p1 ? s_key[xa] : 0ull, kb = xb < p1 ? s_key[xb] : 0ull;
    const uint32_t ha = static_cast<uint32_t>(ka >> 32), hb = static_cast<uint32_t>(kb >> 32);
    const int T4 = (T + 3) & ~3;
    const int span = ((T4 + SR - 1) / SR + 3) & ~3;
    const int u0 = min(T4, sr * span), u1 = min(T4, u0 + span);
    const int m0 = min(max(x0 & ~3, u0), u1), m1 = min(max((x0 + 64 + 3) & ~3, m0), u1);
    const uint4* hh = reinterpret_cast<const uint4*>(s_hi);
    int ca = 0, cb = 0;
#pragma unroll 4
    for (int u = u0; u < m0; u += 4) {   // wholly below x0
      const uint4 h = hh[u >> 2];
      ca += (h.x <= ha) + (h.y <= ha) + (h.z <= ha) + (h.w <= ha);
      cb += (h.x <= hb) + (h.y <= hb) + (h.z <= hb) + (h.w <= hb);
    }
    for (int u = m0; u < m1; ++u) {       // meets x0 .. x0 + 63
      const unsigned long long k = s_key[u];
      ca += k < ka;
      cb += k < kb;
    }
#pragma unroll 4
    for (int u = m1; u < u1; u += 4) {   // wholly at or above x0 + 64
      const uint4 h = hh[u >> 2];
      ca += (h.x < ha) + (h.y < ha) + (h.z < ha) + (h.w < ha);
      cb += (h.x < hb) + (h.y < hb) + (h.z < hb) + (h.w < hb);
    }
    s_part[warp * 64 + lane] = ca;
    s_part[warp * 64 + 32 + lane] = cb;
  }
  __syncthreads();
  // 3. kept flags of this CTA's positions (rank < K), kept counts per warp
  const int li = tid, t = p0 + li;
  const bool own = li < p1 - p0;
  int rank = INT32_MAX;
  if (own) {
    rank = 0;
    for (int sr = 0; sr < SR; ++sr) rank += s_part[sr * G * 64 + li];
    s_rank[li] = rank;
  }
  unsigned ball[kDcutMaxRho];
#pragma unroll
  for (int a = 0; a < kDcutMaxRho; ++a) {
    ball[a] = __ballot_sync(0xffffffffu, a < n_rho && rank < ks.K[a]);
    if (lane == 0 && warp * 32 < P) s_wcnt[warp][a] = __popc(ball[a]);
  }
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every CTA of the cluster runs
  if (tid < n_rho) {   // this CTA's kept count of budget tid, into every CTA
    int c = 0;
    for (int w = 0; w * 32 < P; ++w) c += s_wcnt[w][tid];
    for (uint32_t d = 0; d < kDcCl; ++d) st_cluster_s32(&s_ccnt[crank][tid], d, c);
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");

  // 4. outputs of this CTA's positions: score, keep flags, packing
  if (own) {
    score[t] = __uint_as_float(~s_hi[t]);
    const int r = t / N;
    const bool first = t == r * N;
#pragma unroll
    for (int a = 0; a < kDcutMaxRho; ++a) {
      if (a >= n_rho) break;
      int o = __popc(ball[a] & ((1u << lane) - 1u));   // kept before t: this warp,
      for (int w = 0; w < warp; ++w) o += s_wcnt[w][a];             // earlier warps of the range,
      for (uint32_t c = 0; c < crank; ++c) o += s_ccnt[c][a];       // earlier CTAs
      const bool f = (ball[a] >> lane) & 1u;
      keep[static_cast<int64_t>(a) * T + t] = static_cast<uint8_t>(f);
      if (first && pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + r] = o;
      if (f && pack_idx) pack_idx[static_cast<int64_t>(a) * T + o] = t;
    }
  }
#pragma unroll
  for (int a = 0; a < kDcutMaxRho; ++a) {
    if (a >= n_rho) break;
    const int tot = min(ks.K[a], T);   // rank < K holds for exactly min(K, T) positions
    if (crank == 0 && tid == 0 && pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + B] = tot;
    if (pack_idx)
      for (int q = max(tot, p0) + tid; q < p1; q += kDcutThreads) pack_idx[static_cast<int64_t>(a) * T + q] = -1;
  }
  // keep_len of the requests that start in this CTA's range: one warp per
  // request; ranks past this CTA's range come from the CTAs that hold them
  const int r0 = (p0 + N - 1) / N, r1 = (p1 + N - 1) / N;
  for (int r = r0 + warp; r < r1; r += kDcutThreads / 32) {
    int c[kDcutMaxRho] = {};
    for (int j = lane; j < N; j += 32) {
      const int u = r * N + j;
      const int ou = u / P;
      const int rk = ou == static_cast<int>(crank) ? s_rank[u - p0] : ld_cluster_s32(&s_rank[u - ou * P], ou);
#pragma unroll
      for (int a = 0; a < kDcutMaxRho; ++a) c[a] += a < n_rho && rk < ks.K[a];
    }
#pragma unroll
    for (int a = 0; a < kDcutMaxRho; ++a) {
      if (a < n_rho) {
        const int sum = __reduce_add_sync(0xffffffffu, c[a]);
        if (lane == 0) keep_len[static_cast<int64_t>(a) * B + r] = sum;
      }
    }
  }
  // a request can reach into later CTAs: none may exit while its ranks can be read
  if (P % N != 0) asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Expected tokens per budget: the kept survival probabilities summed exactly
// in fixed point (each score in [0, 1] rounded to a multiple of 2^-50, sums
// of at most 8192 terms fit 64 bits), so the result is within 8192 * 2^-51
// of the exact sum whatever the order; then the budget with the best expected
// tokens per unit of profiled cost.  One CTA of 256 threads: per-thread sums,
// warp sums, then warp 0 adds the 8 warps' (integer sums: any order is exact).
struct DcutCost { float c[kDcutMaxRho]; };
constexpr int kRhoThreads = 256;

__global__ void __launch_bounds__(kRhoThreads) dcut_rho_kernel(const float* __restrict__ score,
                                                               const uint8_t* __restrict__ keep, int T, int n_rho,
                                                               DcutCost cost, double* __restrict__ exp_tok,
                                                               int32_t* __restrict__ rho_star) {
  __shared__ unsigned long long s_acc[kRhoThreads / 32][kDcutMaxRho];
  griddep_wait();
  griddep_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long acc[kDcutMaxRho];
#pragma unroll
  for (int a = 0; a < kDcutMaxRho; ++a) acc[a] = 0ull;
  for (int t = tid; t < T; t += kRhoThreads) {
    const unsigned long long fx = __float2ull_rn(fminf(fmaxf(score[t], 0.f), 1.f) * 0x1p50f);
#pragma unroll
    for (int a = 0; a < kDcutMaxRho; ++a)
      if (a < n_rho && keep[static_cast<int64_t>(a) * T + t]) acc[a] += fx;
  }
#pragma unroll
  for (int a = 0; a < kDcutMaxRho; ++a) {
    unsigned long long v = acc[a];
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_acc[warp][a] = v;
  }
  __syncthreads();
  if (warp != 0) return;
  double best = -1.0;
  int arg = -1;
#pragma unroll
  for (int a = 0; a < kDcutMaxRho; ++a) {
    unsigned long long v = lane < kRhoThreads / 32 ? s_acc[lane][a] : 0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (a < n_rho) {
      const double e = static_cast<double>(v) * 0x1p-50;
      if (lane == 0 && exp_tok) exp_tok[a] = e;
      const double ratio = e / static_cast<double>(cost.c[a]);
      if (ratio > best) { best = ratio; arg = a; }
    }
  }
  if (lane == 0 && rho_star) *rho_star = arg;
}

}  // namespace tv

// The cluster kernel runs unless clusters of 8 full-size CTAs cannot be
// scheduled, or TV_DCUT_PATH=sort asks for the single-CTA sorting network
// (used by the tests to check that path at small T too).
static bool dcut_cluster_ok() {
  static const bool ok = [] {
    const char* e = std::getenv("TV_DCUT_PATH");
    if (e && std::strcmp(e, "sort") == 0) return false;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(tv::kDcCl);
    cfg.blockDim = dim3(tv::kDcutThreads);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tv::dcut_cluster_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    return n > 0;
  }();
  return ok;
}

TV_API size_t dcut_select_workspace_size(int B, int D, int n_rho) {
  (void)B; (void)D; (void)n_rho;
  return 0;
}

TV_API int dcut_select(const float* conf, int B, int D, const float* rho, int n_rho, float* score,
                       uint8_t* keep, int32_t* keep_len, int32_t* pack_off, int32_t* pack_idx,
                       void* ws, size_t ws_bytes, tv_stream_t stream) {
  (void)ws; (void)ws_bytes;
  if (B < 0 || D < 0 || n_rho < 0) return TV_EINVAL;
  if (B == 0 || n_rho == 0) return TV_OK;
  if (n_rho > tv::kDcutMaxRho) return TV_EUNSUPPORTED;
  const long long T = static_cast<long long>(B) * (D + 1);
  if (T > tv::kDcutMaxPos) return TV_EUNSUPPORTED;
  if (!conf && D > 0) return TV_EINVAL;
  if (!rho || !score || !keep || !keep_len) return TV_EINVAL;
  tv::DcutK ks{};
  for (int a = 0; a < n_rho; ++a) {
    const double r = static_cast<double>(rho[a]);   // host array
    if (!(r >= 0.0 && r <= 1.0)) return TV_EINVAL;
    ks.K[a] = static_cast<int>(std::floor(r * static_cast<double>(T) + 0.5));
  }
  const int bytes = tv::kDcutMaxPos * static_cast<int>(sizeof(unsigned long long) + sizeof(int));
  const bool attr = tv::smem_limit(tv::dcut_kernel<1>, bytes) && tv::smem_limit(tv::dcut_kernel<2>, bytes) &&
                    tv::smem_limit(tv::dcut_kernel<4>, bytes) && tv::smem_limit(tv::dcut_kernel<8>, bytes);
  if (!attr) return TV_ECUDA;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  const int Ti = static_cast<int>(T);
  if (Ti <= tv::kDcClMaxT && dcut_cluster_ok())
    return tv::launch_pdl(tv::dcut_cluster_kernel, dim3(tv::kDcCl), dim3(tv::kDcutThreads), 0, st, conf, B, D, n_rho,
                          ks, score, keep, keep_len, pack_off, pack_idx);
  auto kern = Ti <= 1024 ? tv::dcut_kernel<1> : Ti <= 2048 ? tv::dcut_kernel<2> : Ti <= 4096 ? tv::dcut_kernel<4>
                                                                                  : tv::dcut_kernel<8>;
  return tv::launch_pdl(kern, dim3(1), dim3(tv::kDcutThreads), bytes, st, conf, B, D, n_rho, ks, score, keep,
                        keep_len, pack_off, pack_idx);
}

TV_API int dcut_choose_rho(const float* score, const uint8_t* keep, int B, int D, int n_rho, const float* cost,
                           double* exp_tok, int32_t* rho_star, tv_stream_t stream) {
  if (B < 0 || D < 0 || n_rho < 0) return TV_EINVAL;
  if (n_rho > tv::kDcutMaxRho) return TV_EUNSUPPORTED;
  if (B == 0 || n_rho == 0) return TV_OK;
  if (!score || !keep || !cost || (!exp_tok && !rho_star)) return TV_EINVAL;
  const long long T = static_cast<long long>(B) * (D + 1);
  if (T > tv::kDcutMaxPos) return TV_EUNSUPPORTED;
  tv::DcutCost c{};
  for (int a = 0; a < n_rho; ++a) {
    if (!(cost[a] > 0.f)) return TV_EINVAL;   // host array; positive, not NaN
    c.c[a] = cost[a];
  }
  return tv::launch_pdl(tv::dcut_rho_kernel, dim3(1), dim3(tv::kRhoThreads), 0, reinterpret_cast<cudaStream_t>(stream), score,
                        keep, static_cast<int>(T), n_rho, c, exp_tok, rho_star);
}
