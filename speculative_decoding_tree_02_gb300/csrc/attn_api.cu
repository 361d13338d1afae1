// tree_verify_attn entry point: host validation, path choice, workspace
// layout, dispatch.  bf16 with head_dim 128 runs on the tensor cores
// (attn_tc.cu); other shapes (fp32, head_dim 64) on the SIMT path.
#include <cstdlib>
#include <cstring>

#include "attn.cuh"

namespace {


size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// TV_ATTN_PATH=simt forces the SIMT kernels for every shape (used by the
// tests to check both paths on the same inputs); default: by shape.
bool use_tc(int dtype, int d, int Hq, int Hkv) {
  static const int forced = [] {
    const char* e = std::getenv("TV_ATTN_PATH");
    return (e && std::strcmp(e, "simt") == 0) ? 1 : 0;
  }();
  return !forced && tv::attn_tc_supported(dtype, d, Hq, Hkv);
}

struct WsLayout {
  bool tc;
  int n_split;                               // SIMT path
  int piece_len, max_pieces, tiles, n_units;  // tensor-core path
  size_t status, plan, cnt, o_bytes, ml_bytes, total;
};

// SIMT:        [status word (256 B)] [split partials o] [split partials (m, l)]
// tensor core: [status word (256 B)] [work plan] [piece counters]
//              [piece partials o] [piece partials (m, l)]
WsLayout ws_layout(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int d, int dtype) {
  WsLayout w{};
  w.tc = use_tc(dtype, d, Hq, Hkv);
  w.status = 256;
  size_t parts = 0;   // partial rows
  if (w.tc) {
    tv::attn_tc_shape(B, max_nodes, max_prefix, Hq, Hkv, tv::sm_count(), &w.piece_len, &w.max_pieces, &w.tiles);
    w.n_split = 1;
    w.n_units = B * w.tiles * w.max_pieces;   // (request, tile, piece) plan entries
    w.plan = align256(static_cast<size_t>(w.n_units) * sizeof(int4));
    w.cnt = align256(static_cast<size_t>(B) * Hkv * w.tiles * sizeof(int));
    if (w.max_pieces > 1) parts = static_cast<size_t>(w.max_pieces) * B * max_nodes * Hq;
  } else {
    w.n_split = tv::attn_simt_splits(B, max_nodes, max_prefix, Hq, Hkv, tv::sm_count());
    if (w.n_split > 1) parts = static_cast<size_t>(w.n_split) * B * max_nodes * Hq;
  }
  w.o_bytes = align256(parts * d * sizeof(float));
  w.ml_bytes = align256(parts * sizeof(float2));
  w.total = w.status + w.plan + w.cnt + w.o_bytes + w.ml_bytes;
  return w;
}

bool shape_ok(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int d) {
  return B >= 0 && max_nodes >= 0 && max_prefix >= 0 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0 &&
         (d == 64 || d == 128);
}

}  // namespace

TV_API size_t tree_verify_attn_workspace_size(int B, int max_nodes, int max_prefix, int Hq,
                                              int Hkv, int d, int dtype) {
  if (!shape_ok(B, max_nodes, max_prefix, Hq, Hkv, d) || B == 0 || max_nodes == 0) return 0;
  return ws_layout(B, max_nodes, max_prefix, Hq, Hkv, d, dtype).total;
}

TV_API int tree_verify_attn(const void* q, const void* k_pre, const void* v_pre,
                            const int32_t* pre_off, const void* k_tree, const void* v_tree,
                            const int32_t* node_off, const int32_t* node_cnt, const uint64_t* anc,
                            int anc_words, const int32_t* vis_prefix, int B, int max_nodes,
                            int max_prefix, long long total_nodes, long long total_prefix, int Hq,
                            int Hkv, int d, int dtype, float scale, void* out, float* lse,
                            void* ws, size_t ws_bytes, tv_stream_t stream) {
  if (B < 0 || max_nodes < 0 || max_prefix < 0 || Hq <= 0 || Hkv <= 0) return TV_EINVAL;
  if (total_nodes < 0 || total_prefix < 0) return TV_EINVAL;
  if (Hq % Hkv != 0) return TV_EINVAL;
  if (d != 64 && d != 128) return TV_EUNSUPPORTED;
  if (Hq / Hkv > 64) return TV_EUNSUPPORTED;
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_EINVAL;
  if (max_nodes > TV_MAX_NODES) return TV_EUNSUPPORTED;
  if (anc_words < (max_nodes + 63) / 64 || anc_words < 1) return TV_EINVAL;
  if (!(scale > 0.f)) return TV_EINVAL;   // positive and not NaN
  if (B == 0 || max_nodes == 0 || total_nodes == 0) return TV_OK;
  if (max_prefix > total_prefix) return TV_EINVAL;
  if (!q || !pre_off || !k_tree || !v_tree || !node_off || !anc || !out) return TV_EINVAL;
  if (max_prefix > 0 && (!k_pre || !v_pre)) return TV_EINVAL;
  if (static_cast<long long>(B) * Hkv > 65535) return TV_EUNSUPPORTED;
  // 16-byte rows for the vector loads and the tensor maps
  const void* ptrs[] = {q, k_tree, v_tree, out, k_pre, v_pre};
  for (const void* ptr : ptrs)
    if (ptr && !tv::aligned(ptr, 16)) return TV_EINVAL;
  const WsLayout w = ws_layout(B, max_nodes, max_prefix, Hq, Hkv, d, dtype);
  if (!ws || ws_bytes < w.total || !tv::aligned(ws, 256)) return TV_EWORKSPACE;

  tv::AttnParams p{};
  p.q = q; p.k_pre = k_pre; p.v_pre = v_pre; p.pre_off = pre_off;
  p.k_tree = k_tree; p.v_tree = v_tree; p.node_off = node_off; p.node_cnt = node_cnt;
  p.anc = anc; p.vis_prefix = vis_prefix; p.out = out; p.lse = lse;
  p.anc_words = anc_words; p.B = B; p.max_nodes = max_nodes; p.max_prefix = max_prefix;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.dtype = dtype; p.scale = scale; p.n_split = w.n_split;
  char* base = static_cast<char*>(ws);
  char* parts = base + w.status + w.plan + w.cnt;
  if (w.o_bytes) {
    p.ws_o = reinterpret_cast<float*>(parts);
    p.ws_ml = reinterpret_cast<float2*>(parts + w.o_bytes);
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = reinterpret_cast<int*>(base);
  if (w.tc) {   // the planner kernel clears the status word and the counters
    p.plan = reinterpret_cast<const int4*>(base + w.status);
    p.piece_cnt = reinterpret_cast<int*>(base + w.status + w.plan);
    p.piece_len = w.piece_len;
    p.n_units = w.n_units;
    return tv::attn_tc(p, total_nodes, total_prefix, status, st);
  }
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return TV_ECUDA;
  return tv::attn_simt(p, st);
}
