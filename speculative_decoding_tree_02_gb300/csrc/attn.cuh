// Internal interface shared by the tree_verify_attn kernels and its entry point.
#pragma once

#include <algorithm>

#include "tv_common.cuh"

namespace tv {

struct AttnParams {
  const void* q;
  const void* k_pre;
  const void* v_pre;
  const int32_t* pre_off;
  const void* k_tree;
  const void* v_tree;
  const int32_t* node_off;
  const int32_t* node_cnt;
  const uint64_t* anc;
  const int32_t* vis_prefix;
  void* out;
  float* lse;
  float* ws_o;       // [n_split, B*max_nodes, Hq, d] normalised partial outputs
  float2* ws_ml;     // [n_split, B*max_nodes, Hq] (max in log2 units, sum)
  int anc_words;
  int B, max_nodes, max_prefix, Hq, Hkv, d, dtype;
  float scale;
  int n_split;
  // Tensor-core work plan: entry u (grid position z * tiles + y) covers keys
  // [piece * piece_len, (piece + 1) * piece_len) of node tile t of request r,
  // the last piece also the tile's tree keys; the pieces of one (request, KV
  // head, tile) are merged by the last of them to finish.  Entries are
  // ordered longest first.
  const int4* plan;    // [n_units] (r, piece, n_pieces, t); r < 0: no work
  int* piece_cnt;      // [B * Hkv * tiles] finished pieces, zeroed by the planner
  int piece_len;       // keys per piece, a multiple of 64
  int n_units;
};

int attn_simt(const AttnParams& p, cudaStream_t st);
int attn_simt_splits(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int n_sm);
// Merges the key-split partials in split order (shared by both paths).
int attn_combine(const AttnParams& p, cudaStream_t st);

// Tensor-core path: bf16, head_dim 128, Hq/Hkv dividing 128.
bool attn_tc_supported(int dtype, int d, int Hq, int Hkv);
// Piece length and the most pieces per request for a call's sizes (also
// sizes the workspace): requests are split into pieces only when whole
// requests are too few to fill the resident CTAs.
void attn_tc_shape(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int n_sm, int* piece_len,
                   int* max_pieces, int* tiles);
int attn_tc(const AttnParams& p, long long total_nodes, long long total_prefix, int* err, cudaStream_t st);

}  // namespace tv
