// dcut_select: D-cut prefix-product scores and batch-global budget selection
// (D-cut page, technical summary §2 core mechanism and pipeline; §1 B x (D+1)).
//
// One CTA of 1024 threads, everything in shared memory (T = B(D+1) <= 8192):
//   1. one thread per request forms s[r,j] = s[r,j-1] * conf[r,j-1] strictly
//      left to right in fp32 (products only, so nothing can be contracted);
//   2. the T positions are sorted by the 64-bit key (~bits(s), t): scores are
//      non-negative, so their IEEE bits order like the values, and the key
//      order is (s desc, position asc) = (s desc, r asc, j asc).  A bitonic
//      network over the next power of two (padding keys sort last);
//   3. rank(t) = sorted position; t is kept for budget K iff rank(t) < K;
//   4. one block-wide exclusive scan of the keep flags per budget gives the
//      packed slot of every kept position, the per-request offsets and lengths
//      (no assumption that the kept set is a prefix).
#include <cmath>

#include "tv_common.cuh"

namespace tv {

constexpr int kDcutMaxPos = 8192;
constexpr int kDcutMaxRho = 8;
constexpr int kDcutThreads = 1024;

struct DcutK { int K[kDcutMaxRho]; };

// exclusive scan of one int per thread across the 1024-thread block
__device__ __forceinline__ int block_excl_scan(int x, int* s_w, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) s_w[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = s_w[lane];
    int iw = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, iw, o);
      if (lane >= o) iw += y;
    }
    s_w[lane] = iw - w;                 // exclusive warp offsets
    if (lane == 31) s_w[32] = iw;       // block total
  }
  __syncthreads();
  const int r = s_w[warp] + v - x;
  *total = s_w[32];
  __syncthreads();                      // s_w reusable
  return r;
}

__global__ void __launch_bounds__(kDcutThreads) dcut_kernel(
    const float* __restrict__ conf, int B, int D, int n_rho, DcutK ks, float* __restrict__ score,
    uint8_t* __restrict__ keep, int32_t* __restrict__ keep_len, int32_t* __restrict__ pack_off,
    int32_t* __restrict__ pack_idx) {
  extern __shared__ unsigned long long s_key[];                       // [Tp] sort keys
  int* s_rank = reinterpret_cast<int*>(s_key + kDcutMaxPos);          // [T]
  __shared__ int s_w[33];
  const int tid = threadIdx.x;
  const int N = D + 1;
  const int T = B * N;
  int Tp = 1;
  while (Tp < T) Tp <<= 1;

  // 1. scores, and their sort keys
  for (int r = tid; r < B; r += blockDim.x) {
    float s = 1.f;
    for (int j = 0; j <= D; ++j) {
      if (j > 0) s = __fmul_rn(s, conf[static_cast<int64_t>(r) * D + j - 1]);
      const int t = r * N + j;
      score[t] = s;
      s_key[t] = (static_cast<unsigned long long>(~__float_as_uint(s)) << 32) | static_cast<unsigned>(t);
    }
  }
  for (int t = T + tid; t < Tp; t += blockDim.x) s_key[t] = ~0ull;
  __syncthreads();

  // 2. bitonic sort, ascending keys
  for (int k = 2; k <= Tp; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < Tp; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const unsigned long long a = s_key[i], b = s_key[p];
          const bool up = (i & k) == 0;
          if ((a > b) == up) { s_key[i] = b; s_key[p] = a; }
        }
      }
      __syncthreads();
    }
  }
  // 3. rank of each position
  for (int i = tid; i < T; i += blockDim.x) s_rank[static_cast<int>(s_key[i] & 0xffffffffu)] = i;
  __syncthreads();

  // 4. per budget: flags, exclusive scan, packing
  const int per = (T + blockDim.x - 1) / blockDim.x;     // consecutive positions per thread
  const int t0 = tid * per;
  for (int a = 0; a < n_rho; ++a) {
    const int K = ks.K[a];
    uint8_t* kp = keep + static_cast<int64_t>(a) * T;
    int mine = 0;
    for (int t = t0; t < min(T, t0 + per); ++t) {
      const int f = s_rank[t] < K;
      kp[t] = static_cast<uint8_t>(f);
      mine += f;
    }
    int total = 0;
    int o = block_excl_scan(mine, s_w, &total);
    int32_t* pi = pack_idx ? pack_idx + static_cast<int64_t>(a) * T : nullptr;
    for (int t = t0; t < min(T, t0 + per); ++t) {
      const int f = s_rank[t] < K;
      const int r = t / N, j = t - r * N;
      if (j == 0 && pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + r] = o;   // kept before request r
      if (f && pi) pi[o] = t;
      o += f;
    }
    if (tid == 0 && pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + B] = total;
    if (pi)
      for (int q = total + tid; q < T; q += blockDim.x) pi[q] = -1;
    // keep_len[r] = kept positions of request r
    for (int r = tid; r < B; r += blockDim.x) {
      int c = 0;
      for (int j = 0; j < N; ++j) c += s_rank[r * N + j] < K;
      keep_len[static_cast<int64_t>(a) * B + r] = c;
    }
  }
}

}  // namespace tv

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
  static const int smem = [] {
    const int bytes = tv::kDcutMaxPos * static_cast<int>(sizeof(unsigned long long) + sizeof(int));
    cudaFuncSetAttribute(tv::dcut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return bytes;
  }();
  tv::dcut_kernel<<<1, tv::kDcutThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      conf, B, D, n_rho, ks, score, keep, keep_len, pack_off, pack_idx);
  return tv::launch_status();
}
