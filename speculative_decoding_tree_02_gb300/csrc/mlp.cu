// blockpilot_mlp: BlockPilot's block-size predictor (BlockPilot page §3: the
// last-prefill next-token distribution feeds a two-layer MLP that picks the
// block size once per request; §7 raw probabilities as input; §4 hidden 2048;
// §2 candidates B-3 .. B+3).
//
// Layer 1, up to 8 requests (tensor cores): D[h, c] = sum_v W1[v, h] X[c, v]
// with tcgen05 MMAs, M = 128 hidden units per CTA, N = 16: X rows 0..7 are
// the probabilities rounded to bf16 (x_hi), rows 8..15 the rounding
// remainders (x_lo = bf16(x - x_hi)), so h = D[., b] + D[., 8 + b] carries x
// to about 16 mantissa bits.  W1 streams through a TMA ring once (split-K
// over V across CTAs); its tile is the MN-major A operand, X the K-major B.
// The same kernel finishes the job: the last K split of each hidden tile
// reduces the tile's partials and forms its share of layer 2, the last tile
// adds the shares and takes the argmax.
//
// Fallback layer 1 (more requests): a bandwidth-bound GEMV with 8 right-hand sides (the requests):
// every W1 element is read once and used for 8 FMAs.  Grid (column block of
// 256 hidden units, V-slice, request group of 8).  The softmax is fused: the
// CTA first turns its slice of each request's logits into probabilities
// x = 2^((l - lse) log2 e) in shared memory.  Warps take W1 rows round-robin,
// lanes own 8 hidden units (one 16-byte load per row), and the 8 warps'
// partial sums are reduced through shared memory in warp order.  Layer 2,
// ReLU and the argmax then run in one small CTA per request, summing the
// V-slices in slice order (deterministic).
#include <algorithm>
#include <cstring>

#include "tc_common.cuh"

namespace tv {

constexpr int kMThreads = 256;
constexpr int kMCols = 256;        // hidden units per CTA (8 per lane, 32 lanes)
constexpr int kMReq = 8;           // requests per CTA
constexpr int kMSub = 256;         // rows of x staged at a time

__global__ void __launch_bounds__(kMThreads) mlp_l1_kernel(
    const uint16_t* __restrict__ logits, int64_t ld, const float* __restrict__ row_lse,
    const uint16_t* __restrict__ W1, int B, int V, int H, int rows_per_slice,
    float* __restrict__ part) {
  __shared__ __align__(16) float s_x[kMSub][kMReq];
  __shared__ float s_red[kMThreads / 32][kMCols];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cb = blockIdx.x, slice = blockIdx.y, rg = blockIdx.z;
  const int v0 = slice * rows_per_slice;
  const int v1 = min(V, v0 + rows_per_slice);
  const int nb = min(kMReq, B - rg * kMReq);
  const int col0 = cb * kMCols + lane * 8;

  float acc[kMReq][8];
#pragma unroll
  for (int b = 0; b < kMReq; ++b)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[b][c] = 0.f;

  for (int s0 = v0; s0 < v1; s0 += kMSub) {
    __syncthreads();
    {
      const int v = s0 + tid;
#pragma unroll
      for (int b = 0; b < kMReq; ++b) {
        float x = 0.f;
        if (b < nb && v < v1) {
          const int rq = rg * kMReq + b;
          const float l = bf16_at(logits + static_cast<int64_t>(rq) * ld + v);
          x = ex2(fmaf(l, kLog2e, -row_lse[rq] * kLog2e));
        }
        s_x[tid][b] = x;
      }
    }
    __syncthreads();
    const int n = min(kMSub, v1 - s0);
    for (int j = warp; j < n; j += kMThreads / 32) {
      const uint4 w = ldg_stream(W1 + static_cast<int64_t>(s0 + j) * H + col0);
      const float wf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                           bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
      const float4 xa = *reinterpret_cast<const float4*>(&s_x[j][0]);
      const float4 xb = *reinterpret_cast<const float4*>(&s_x[j][4]);
      const float xs[kMReq] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int b = 0; b < kMReq; ++b)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[b][c] = fmaf(xs[b], wf[c], acc[b][c]);
    }
  }
  // reduce the 8 warps' partials, one request at a time, in warp order
  for (int b = 0; b < nb; ++b) {
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 8; ++c) s_red[warp][lane * 8 + c] = acc[b][c];
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kMThreads / 32; ++w) t += s_red[w][tid];
    const int rq = rg * kMReq + b;
    part[(static_cast<int64_t>(slice) * B + rq) * H + cb * kMCols + tid] = t;
  }
}

__global__ void __launch_bounds__(256) mlp_l2_kernel(
    const float* __restrict__ part, int n_slice, int B, int H, int C,
    const float* __restrict__ b1, const uint16_t* __restrict__ W2, const float* __restrict__ b2,
    int block, float* __restrict__ z, int32_t* __restrict__ choice, int32_t* __restrict__ bsize) {
  __shared__ float s_z[256 / 32][32];
  griddep_wait();
  griddep_release();
  const int rq = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float zc[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) zc[c] = 0.f;
  for (int h = tid; h < H; h += blockDim.x) {
    float a = b1 ? b1[h] : 0.f;
    for (int s = 0; s < n_slice; ++s) a += part[(static_cast<int64_t>(s) * B + rq) * H + h];
    a = fmaxf(a, 0.f);
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (c < C) zc[c] = fmaf(a, bf16_at(W2 + static_cast<int64_t>(h) * C + c), zc[c]);
  }
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float v = warp_sum(zc[c]);
    if (lane == 0) s_z[warp][c] = v;
  }
  __syncthreads();
  if (tid == 0) {
    int best = 0;
    float bv = -INFINITY;
    for (int c = 0; c < C; ++c) {
      float v = b2 ? b2[c] : 0.f;
      for (int w = 0; w < 256 / 32; ++w) v += s_z[w][c];
      z[static_cast<int64_t>(rq) * C + c] = v;
      if (v > bv) { bv = v; best = c; }
    }
    choice[rq] = best;
    bsize[rq] = block - (C - 1) / 2 + best;
  }
}

// ------------------------------------------------------------ tensor-core layer 1
constexpr int kQTile = 128;                        // hidden units per CTA (MMA M)
constexpr int kQK = 64;                            // v per pipeline stage (four K = 16 MMAs)
constexpr int kQN = 16;                            // x_hi rows 0..7, x_lo rows 8..15 (MMA N)
constexpr int kQStages = 6;
constexpr int kQCtas = 2;        // CTAs per SM
constexpr int kQThreads = 192;                     // TMA warp, MMA warp, 4 epilogue warps
constexpr uint32_t kQAHalf = 64 * kQK * 2;         // 64 hidden x 64 v, bf16: 8 KB
constexpr uint32_t kQStageBytes = 2 * kQAHalf + kQN * kQK * 2;   // 16 KB + 2 KB
constexpr uint32_t kQBarOff = kQStages * kQStageBytes;
constexpr uint32_t kQSmem = kQBarOff + 256 + 1024;  // barriers, TMEM slot, status; 1 KB alignment slack
constexpr size_t kMlpHdrBytes = 256;               // workspace: status word, then X, then partials

struct MlpMaps { CUtensorMap w1, x; };
struct MlpTcParams {
  MlpMaps maps;
  int H, B, C, block, ksteps, kps;
  float* part;          // [splits][B][H] layer-1 partial sums
  int* err;
  int* cnt;             // [tiles + 1] arrival counters, zero between calls
  float* zpart;         // [tiles][B][C] layer-2 partial sums
  const float* b1;
  const uint16_t* W2;
  const float* b2;
  float* z;
  int32_t* choice;
  int32_t* bsize;
};

// x = softmax(logits) rows as bf16 hi/lo pairs: X[c][v], c < 8 hi, c >= 8 lo;
// rows of absent requests are zero.  Also clears the status word and the
// layer-1 kernel's arrival counters.
__global__ void __launch_bounds__(256) mlp_x_kernel(const uint16_t* __restrict__ logits, int64_t ld,
                                                    const float* __restrict__ row_lse, int B, int V, int Vp,
                                                    uint16_t* __restrict__ X, int* __restrict__ err,
                                                    int* __restrict__ cnt, int n_cnt) {
  griddep_wait();
  griddep_release();
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v == 0 && err) *err = 0;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
  if (v >= V) return;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    uint16_t hi = 0, lo = 0;
    if (b < B) {
      const float l = bf16_at(logits + static_cast<int64_t>(b) * ld + v);
      const float x = ex2(fmaf(l, kLog2e, -row_lse[b] * kLog2e));
      const __nv_bfloat16 h = __float2bfloat16_rn(x);
      const __nv_bfloat16 r = __float2bfloat16_rn(x - __bfloat162float(h));
      hi = *reinterpret_cast<const uint16_t*>(&h);
      lo = *reinterpret_cast<const uint16_t*>(&r);
    }
    X[static_cast<int64_t>(b) * Vp + v] = hi;
    X[static_cast<int64_t>(8 + b) * Vp + v] = lo;
  }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// CTA (hidden tile, K split).  Every wait is bounded; on expiry the CTA
// records an error code in the status word, stops, and releases its TMEM.
// Tail: the last split of a hidden tile to finish (arrival counter) sums the
// tile's partials in split order, adds b1, applies the ReLU and forms the
// tile's share of layer 2; the last tile to finish sums those shares in tile
// order, adds b2 and takes the argmax.  Both orders are fixed, so the result
// does not depend on which CTA happens to arrive last.
__global__ void __launch_bounds__(kQThreads, kQCtas) mlp_tc_kernel(const __grid_constant__ MlpTcParams P) {
  using namespace tc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ht = blockIdx.x, split = blockIdx.y;
  const int k0 = split * P.kps, n = max(0, min(P.ksteps, k0 + P.kps) - k0);
  auto full = [&](int s) { return sb + kQBarOff + 8u * s; };
  auto empty = [&](int s) { return sb + kQBarOff + 8u * (kQStages + s); };
  const uint32_t done = sb + kQBarOff + 8u * (2 * kQStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kQBarOff + 8 * (2 * kQStages + 1) + 4);
  // Warp 0 (the TMA producer) waits for the softmax kernel later, after its
  // first W1 loads: W1 is an input of the call, and the softmax kernel lets
  // this grid launch only after its own wait on whatever ran before the call.
  if (warp != 0) griddep_wait();
  griddep_release();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    mbar_init(done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const uint32_t tslot = sb + kQBarOff + 8 * (2 * kQStages + 1);
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(tslot) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kQBarOff + 8 * (2 * kQStages + 1));
  int* err = P.err;

  if (warp == 0) {
    if (lane == 0) {   // ================= TMA producer
      // the first ring's W1 tiles go out while the softmax kernel may still run
      const int pre = min(n, kQStages);
      for (int i = 0; i < pre; ++i) {
        const uint32_t dst = sb + i * kQStageBytes;
        const int v = (k0 + i) * kQK;
        mbar_expect_tx(full(i), kQStageBytes);
        tma_load_2d(dst, &P.maps.w1, ht * kQTile, v, full(i));
        tma_load_2d(dst + kQAHalf, &P.maps.w1, ht * kQTile + 64, v, full(i));
      }
      griddep_wait();
      for (int i = 0; i < pre; ++i)
        tma_load_2d(sb + i * kQStageBytes + 2 * kQAHalf, &P.maps.x, (k0 + i) * kQK, 0, full(i));
      for (int i = pre; i < n; ++i) {
        const int s = i % kQStages;
        if (!mbar_wait(empty(s), ((i / kQStages) - 1) & 1, abort_flag, err, 21)) break;
        const uint32_t dst = sb + s * kQStageBytes;
        const int v = (k0 + i) * kQK;
        mbar_expect_tx(full(s), kQStageBytes);
        tma_load_2d(dst, &P.maps.w1, ht * kQTile, v, full(s));
        tma_load_2d(dst + kQAHalf, &P.maps.w1, ht * kQTile + 64, v, full(s));
        tma_load_2d(dst + 2 * kQAHalf, &P.maps.x, v, 0, full(s));
      }
    }
    __syncwarp();
    griddep_wait();
  } else if (warp == 1) {
    if (lane == 0) {   // ================= MMA issuer
      // M = 128, N = 16, A MN-major (transpose bit 15), B K-major
      constexpr uint32_t idesc = idesc_bf16(kQTile, kQN, 0) | (1u << 15);
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const int s = i % kQStages;
        ok = mbar_wait(full(s), (i / kQStages) & 1, abort_flag, err, 22);
        if (!ok) break;
        tc_fence_after();
        const uint32_t abase = sb + s * kQStageBytes, bbase = abase + 2 * kQAHalf;
#pragma unroll
        for (int kk = 0; kk < kQK / 16; ++kk)
          umma_bf16(tmem, sdesc(abase + kk * 2048, kQAHalf, 1024), sdesc(bbase + kk * 32, 16, 1024), idesc,
                    (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(empty(s));
      }
      if (n > 0) umma_commit(done);
      else mbar_arrive(done);
    }
  } else {   // ================= epilogue: D rows of this warp's TMEM lane quarter
    const bool ok = mbar_wait(done, 0, abort_flag, err, 23);
    tc_fence_after();
    uint32_t d[16];
    tmem_ld16(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16), d);
    tmem_ld_wait();
    const int h = ht * kQTile + 32 * (warp & 3) + lane;
    if (ok) {
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (b >= P.B) break;
        const float v = n > 0 ? __uint_as_float(d[b]) + __uint_as_float(d[8 + b]) : 0.f;
        P.part[(static_cast<int64_t>(split) * P.B + b) * P.H + h] = v;
      }
    }
    __threadfence();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem) : "memory");
  }

  // ---------------- tail: split-K reduction, ReLU, layer 2, argmax
  const int tiles = gridDim.x, splits = gridDim.y;
  volatile int* s_flag = reinterpret_cast<volatile int*>(sm + kQBarOff + 8 * (2 * kQStages + 2));
  if (threadIdx.x == 0) *s_flag = atomicAdd(&P.cnt[ht], 1) == splits - 1;
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  if (threadIdx.x == 0) P.cnt[ht] = 0;
  // The ring is free (every MMA has completed): stage 0 holds the tile's W2
  // rows (128 x C bf16, contiguous in W2) and, later, the layer-2 shares.
  uint16_t* s_w2 = reinterpret_cast<uint16_t*>(sm);
  float* s_z = reinterpret_cast<float*>(sm + 8192);              // [B][C]
  float* s_zp = reinterpret_cast<float*>(sm + 8192 + 1024);      // [tiles][B][C]
  {
    const uint16_t* src = P.W2 + static_cast<int64_t>(ht) * kQTile * P.C;
#pragma unroll 8
    for (int i = threadIdx.x; i < kQTile * P.C; i += blockDim.x) s_w2[i] = src[i];
  }
  // lane q owns hidden units 4q .. 4q+3 of the tile; warp w < 4 requests w and w + 4
  const int q = lane, h0 = ht * kQTile + 4 * q;
  const int rb0 = warp, rb1 = warp + 4;
  const bool has0 = warp < 4 && rb0 < P.B, has1 = warp < 4 && rb1 < P.B;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (warp < 4 && P.b1) a0 = *reinterpret_cast<const float4*>(P.b1 + h0);
  float4 a1 = a0;
  {
    const int64_t sstride = static_cast<int64_t>(P.B) * P.H;
    const float* p0 = P.part + static_cast<int64_t>(rb0) * P.H + h0;
    const float* p1 = P.part + static_cast<int64_t>(rb1) * P.H + h0;
#pragma unroll 8
    for (int s = 0; s < splits; ++s) {   // split order
      if (has0) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(p0 + s * sstride));
        a0.x += t.x; a0.y += t.y; a0.z += t.z; a0.w += t.w;
      }
      if (has1) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(p1 + s * sstride));
        a1.x += t.x; a1.y += t.y; a1.z += t.z; a1.w += t.w;
      }
    }
  }
  __syncthreads();   // W2 rows staged
  if (warp < 4) {
    const float r0[4] = {fmaxf(a0.x, 0.f), fmaxf(a0.y, 0.f), fmaxf(a0.z, 0.f), fmaxf(a0.w, 0.f)};
    const float r1[4] = {fmaxf(a1.x, 0.f), fmaxf(a1.y, 0.f), fmaxf(a1.z, 0.f), fmaxf(a1.w, 0.f)};
    for (int c = 0; c < P.C; ++c) {
      float z0 = 0.f, z1 = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float w = __uint_as_float(static_cast<uint32_t>(s_w2[(4 * q + i) * P.C + c]) << 16);
        z0 = fmaf(r0[i], w, z0);
        z1 = fmaf(r1[i], w, z1);
      }
      z0 = warp_sum(z0);
      z1 = warp_sum(z1);
      if (q == 0 && has0) P.zpart[(static_cast<int64_t>(ht) * P.B + rb0) * P.C + c] = z0;
      if (q == 0 && has1) P.zpart[(static_cast<int64_t>(ht) * P.B + rb1) * P.C + c] = z1;
    }
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) *s_flag = atomicAdd(&P.cnt[tiles], 1) == tiles - 1;
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  if (threadIdx.x == 0) P.cnt[tiles] = 0;
  const int n_zp = tiles * P.B * P.C;
  const bool staged = static_cast<uint32_t>(n_zp) * 4u <= kQBarOff - 8192u - 1024u;
  if (staged) {
#pragma unroll 4
    for (int i = threadIdx.x; i < n_zp; i += blockDim.x) s_zp[i] = __ldcg(P.zpart + i);
    __syncthreads();
  }
  for (int i = threadIdx.x; i < P.B * P.C; i += blockDim.x) {
    const int b = i / P.C, c = i - b * P.C;
    float v = P.b2 ? P.b2[c] : 0.f;
    for (int t = 0; t < tiles; ++t) {   // tile order
      const int64_t j = (static_cast<int64_t>(t) * P.B + b) * P.C + c;
      v += staged ? s_zp[j] : __ldcg(P.zpart + j);
    }
    P.z[i] = v;
    s_z[i] = v;
  }
  __syncthreads();
  if (threadIdx.x < P.B) {
    const int b = threadIdx.x;
    int best = 0;
    float bv = -INFINITY;
    for (int c = 0; c < P.C; ++c)
      if (s_z[b * P.C + c] > bv) { bv = s_z[b * P.C + c]; best = c; }
    P.choice[b] = best;
    P.bsize[b] = P.block - (P.C - 1) / 2 + best;
  }
}

static bool mlp_map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_in, uint32_t box_out) {
  auto enc = tc::encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_in, box_out};
  cuuint32_t estr[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// tensor-core path geometry: K splits so that (H / 128) x splits fill kQCtas CTAs per SM
static void mlp_tc_shape(int V, int H, int n_sm, int* ksteps, int* kps, int* splits) {
  *ksteps = (V + kQK - 1) / kQK;
  const int tiles = H / kQTile;
  int s = std::max(1, (kQCtas * n_sm + tiles - 1) / tiles);
  s = std::min(s, *ksteps);
  *kps = (*ksteps + s - 1) / s;
  *splits = (*ksteps + *kps - 1) / *kps;
}

// counters (tiles + 1, padded to 256 B) and layer-2 partials (tiles x B x 32) after the partials
static size_t mlp_cnt_bytes(int H) { return (static_cast<size_t>(H / kQTile + 1) * sizeof(int) + 255) / 256 * 256; }
static size_t mlp_tail_bytes(int B, int H) {
  return mlp_cnt_bytes(H) + static_cast<size_t>(H / kQTile) * B * 32 * sizeof(float);
}

static bool mlp_tc_ok(int B, int V, int H, int64_t ld, const void* W1, const float* b1) {
  return B <= 8 && H % kQTile == 0 && (static_cast<int64_t>(H) * 2) % 16 == 0 && aligned(W1, 16) &&
         (!b1 || aligned(b1, 16)) && V >= 1 && ld >= V;
}

int mlp_slices(int V, int H, int B) {
  const int n_sm = sm_count();
  const int ctas_per_slice = (H / kMCols) * ((B + kMReq - 1) / kMReq);
  int s = (4 * n_sm + ctas_per_slice - 1) / ctas_per_slice;
  s = std::max(1, std::min(s, (V + kMSub - 1) / kMSub));
  return s;
}

}  // namespace tv


TV_API size_t blockpilot_mlp_workspace_size(int B, int V, int H) {
  if (B <= 0 || V <= 0 || H <= 0) return 0;
  const size_t simt = static_cast<size_t>(tv::mlp_slices(V, H, B)) * B * H * sizeof(float);
  int ksteps = 0, kps = 0, splits = 0;
  tv::mlp_tc_shape(V, H, tv::sm_count(), &ksteps, &kps, &splits);
  const size_t Vp = (static_cast<size_t>(V) + 63) / 64 * 64;
  const size_t tcb = tv::kMlpHdrBytes + 16 * Vp * 2 + static_cast<size_t>(splits) * B * H * sizeof(float) +
                     tv::mlp_tail_bytes(B, H);
  return std::max(simt, tcb);
}

TV_API int blockpilot_mlp(const void* last_logits, int64_t ld, const float* row_lse,
                          const void* W1, const float* b1, const void* W2, const float* b2, int B,
                          int V, int H, int C, int block, float* z, int32_t* choice,
                          int32_t* bsize, void* ws, size_t ws_bytes, tv_stream_t stream) {
  if (B < 0 || V <= 0 || H <= 0 || C <= 0 || ld < V) return TV_EINVAL;
  if (H % tv::kMCols != 0 || C > 32 || B > 16) return TV_EUNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!last_logits || !row_lse || !W1 || !W2 || !z || !choice || !bsize) return TV_EINVAL;
  if (!tv::aligned(W1, 16)) return TV_EINVAL;
  const size_t need = blockpilot_mlp_workspace_size(B, V, H);
  if (!ws || ws_bytes < need || !tv::aligned(ws, 16)) return TV_EWORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (tv::mlp_tc_ok(B, V, H, ld, W1, b1)) {
    int ksteps = 0, kps = 0, splits = 0;
    tv::mlp_tc_shape(V, H, tv::sm_count(), &ksteps, &kps, &splits);
    const int Vp = (V + 63) / 64 * 64;
    char* base = static_cast<char*>(ws);
    int* err = reinterpret_cast<int*>(base);
    auto* X = reinterpret_cast<uint16_t*>(base + tv::kMlpHdrBytes);
    auto* part = reinterpret_cast<float*>(base + tv::kMlpHdrBytes + static_cast<size_t>(16) * Vp * 2);
    tv::MlpTcParams P;
    std::memset(&P, 0, sizeof(P));
    if (!tv::mlp_map2d(&P.maps.w1, W1, static_cast<uint64_t>(H), static_cast<uint64_t>(V),
                       static_cast<uint64_t>(H) * 2, 64, tv::kQK) ||
        !tv::mlp_map2d(&P.maps.x, X, static_cast<uint64_t>(V), 16, static_cast<uint64_t>(Vp) * 2, tv::kQK, 16))
      return TV_ECUDA;
    const int tiles = H / tv::kQTile;
    int* cnt = reinterpret_cast<int*>(reinterpret_cast<char*>(part) + static_cast<size_t>(splits) * B * H * 4);
    P.H = H; P.B = B; P.C = C; P.block = block; P.ksteps = ksteps; P.kps = kps; P.part = part; P.err = err;
    P.cnt = cnt;
    P.zpart = reinterpret_cast<float*>(reinterpret_cast<char*>(cnt) + tv::mlp_cnt_bytes(H));
    P.b1 = b1; P.W2 = static_cast<const uint16_t*>(W2); P.b2 = b2;
    P.z = z; P.choice = choice; P.bsize = bsize;
    if (!tv::smem_limit(tv::mlp_tc_kernel, static_cast<int>(tv::kQSmem))) return TV_ECUDA;
    int rc = tv::launch_pdl(tv::mlp_x_kernel, dim3((V + 255) / 256), dim3(256), 0, st,
                            static_cast<const uint16_t*>(last_logits), ld, row_lse, B, V, Vp, X, err, cnt,
                            tiles + 1);
    if (rc == TV_OK)
      rc = tv::launch_pdl(tv::mlp_tc_kernel, dim3(tiles, splits), dim3(tv::kQThreads), tv::kQSmem, st, P);
    return rc;
  }
  const int n_slice = tv::mlp_slices(V, H, B);
  const int rows_per_slice = (V + n_slice - 1) / n_slice;
  dim3 g1(H / tv::kMCols, n_slice, (B + tv::kMReq - 1) / tv::kMReq);
  tv::mlp_l1_kernel<<<g1, tv::kMThreads, 0, st>>>(
      static_cast<const uint16_t*>(last_logits), ld, row_lse, static_cast<const uint16_t*>(W1), B,
      V, H, rows_per_slice, static_cast<float*>(ws));
  tv::mlp_l2_kernel<<<B, 256, 0, st>>>(static_cast<const float*>(ws), n_slice, B, H, C, b1,
                                       static_cast<const uint16_t*>(W2), b2, block, z, choice,
                                       bsize);
  return tv::launch_status();
}
