// Argument blocks and launchers of the libsa27 kernels (internal header).
#pragma once
#include "common.cuh"

namespace sa {

struct CompressArgs {
  int dtype, ik_dtype, B, d, dI, m;
  const void* k_raw;
  const void* v_raw;
  const void* ik_raw;
  const float* z;
  int R;
  const int32_t* blk_lo;
  const int32_t* blk_hi;
  int max_blocks;
  void* k_c;
  void* v_c;
  void* ik_c;
  void* ik_c_scales;
  int N_cap;
  int32_t* err;
};
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t st);
cudaError_t launch_mxfp4_quantize(const void* x_bf16, int64_t nblk, void* codes, void* scales,
                                  cudaStream_t st);

// Indexer scoring: scores[r*ld + j] for j < n(r) = min(N_cap, (q_pos[r]+1)/m).
struct ScoreArgs {
  int dtype, B, T, HI, dI, m;
  const void* q;        // [B*T, HI, dI] (MXFP4: codes [.., dI/2])
  const void* q_scales; // MXFP4 only: [B*T, HI, dI/32]
  const float* w;       // [B*T, HI]
  const void* ik;       // [B, N_cap, dI] (MXFP4: codes)
  const void* ik_scales;
  int N_cap;
  const int32_t* q_pos;
  float* scores;
  int64_t ld;
  int32_t* err;
};
cudaError_t launch_score_simt(const ScoreArgs& a, cudaStream_t st);
cudaError_t launch_score_tc(const ScoreArgs& a, int num_sms, cudaStream_t st);
bool score_tc_supported(const ScoreArgs& a);
cudaError_t launch_score_mx(const ScoreArgs& a, int num_sms, cudaStream_t st);
bool score_mx_supported(const ScoreArgs& a);

// Per-row top-k over scores (see csa_index_topk).
struct TopkArgs {
  const float* scores;
  int64_t ld;
  const int32_t* q_pos;
  int rows, m, N_cap, k;
  int32_t* idx;
  int32_t* err;
};
cudaError_t launch_topk(const TopkArgs& a, int num_sms, cudaStream_t st);
bool topk_supported(int N_cap);

// Attention over (compressed part) + (window part) per query row.
//  Compressed part: gathered (gather = 1: idx slots [0, min(k, n)), n = (p+1)/m,
//  entries -1 skipped) or dense (gather = 0: rows [0, n)).
//  Window part: raw positions p-Wn+1 .. p in ring rows (u mod R).
struct AttnArgs {
  int dtype, B, T, H, d;
  float sm_scale;
  const void* q;        // [B*T, H, d]
  const int32_t* q_pos;
  const void* kc;       // [B, N_cap, d]
  const void* vc;
  int N_cap;
  const int32_t* idx;   // [B*T, k] when gather
  int gather;           // 1: CSA (idx slots), 0: dense compressed rows (HCA)
  int k, m;
  const void* kr;       // [B, R, d]
  const void* vr;
  int R, W;
  void* o;              // [B*T, H, d] in o_dtype
  int o_dtype;          // SA_F32 or SA_BF16
  float* lse;           // [B*T, H]
  int nsplit;           // key-tile splits per row (1: write o/lse directly)
  int split_tiles;      // key tiles (of kAttnTile keys) per split
  float* part_o;        // [B*T, nsplit, H, d] when nsplit > 1
  float* part_lse;      // [B*T, nsplit, H]
  unsigned* item_counter;   // zeroed before the launch: items taken dynamically (or NULL)
  int32_t* err;
};
constexpr int kAttnTile = 64;     // keys per attention tile (split granularity)
// tensor-core kernel: key tiles per split at most (a loop bound only: the
// running sums stay below 2^32 per key, far inside fp32, at any length)
constexpr int kAttnTcMaxSplitTiles = 1 << 16;
cudaError_t launch_attend_simt(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_attend_tc(const AttnArgs& a, int num_sms, cudaStream_t st);
bool attend_tc_supported(const AttnArgs& a);
int attend_tc_items_per_sm();   // (row, split) items per SM the split choice aims at
// Merge nsplit partials per (row, head) into o/lse.
cudaError_t launch_merge_splits(const AttnArgs& a, cudaStream_t st);

// Fused CSA decode (csa_decode): one cluster of C CTAs per sequence, one
// query token each.  All tensors bf16 unless stated.
struct FusedDecodeArgs {
  int B, H, m, k, W;
  float sm_scale;
  const void* q;        // [B, H, 128]
  const void* q_idx;    // [B, 64, 64]
  const float* w;       // [B, 64] f32
  const int32_t* q_pos; // [B]
  const void* k_raw;    // [B, R, 128]
  const void* v_raw;
  const void* ik_raw;   // [B, R, 64]
  const float* z;       // [B, R] f32
  int R;
  const int32_t* blk_lo;
  const int32_t* blk_hi;
  int max_blocks;
  void* k_c;            // [B, N_cap, 128] (blocks [blk_lo, blk_hi) written)
  void* v_c;
  void* ik_c;           // [B, N_cap, 64]
  int N_cap;
  int32_t* idx;         // [B, k] int32
  void* o;              // [B, H, 128] in o_dtype
  int o_dtype;
  float* lse;           // [B, H] f32
  int32_t* err;
  // launch plan (fused_decode_plan)
  int C;                // CTAs per cluster (one cluster per sequence)
  int cap;              // key slots per CTA (8192 or 16384)
  int selcap;           // selected-list slots per CTA
  int stages_a;         // indexer-key stages (16 KB)
  int stages_kv;        // K/V stages (32 KB)
};
bool fused_decode_plan(FusedDecodeArgs& a, int num_sms);
cudaError_t launch_fused_decode(const FusedDecodeArgs& a, cudaStream_t st);

// sa_compress_channels: per-channel softmax pooling of one array.
struct CompressChArgs {
  int dtype, B, d, m, R, max_blocks, N_cap;
  const void* x_raw;    // [B, R, d]
  const float* z;       // [B, R, d] f32
  const int32_t* blk_lo;
  const int32_t* blk_hi;
  void* x_c;            // [B, N_cap, d]
  int32_t* err;
};
cudaError_t launch_compress_channels(const CompressChArgs& a, cudaStream_t st);

// sa_ring_write: row b of array i into ring i's row pos[b] mod R.
constexpr int kRingMaxArrays = 8;
struct RingWriteArgs {
  int B, R, n;
  const int32_t* pos;
  void* rings[kRingMaxArrays];
  const void* rows[kRingMaxArrays];
  int row_bytes[kRingMaxArrays];
  int32_t* err;
};
cudaError_t launch_ring_write(const RingWriteArgs& a, cudaStream_t st);

// Whole hybrid decode step (sa_decode_step): both layers of one decode token
// per sequence in one persistent launch over a queue of work items.  All
// tensors bf16 unless stated.
constexpr int kStepMaxTilesPerPart = 32;   // key tiles per attention share at most
struct StepArgs {
  int B, H, m, k, W, m2;
  float sm_scale;
  const void* q;        // [B, H, 128] CSA queries
  const void* q_idx;    // [B, 64, 64]
  const float* w;       // [B, 64] f32
  const void* q_hca;    // [B, H, 128] HCA queries
  const int32_t* q_pos; // [B]
  const void* k_raw;    // [B, R, 128]
  const void* v_raw;
  const void* ik_raw;   // [B, R, 64]
  const float* z;       // [B, R] f32
  const void* hk_raw;   // [B, R, 128]
  const void* hv_raw;
  const float* hz;      // [B, R] f32
  int R;
  const int32_t* blk_lo;
  const int32_t* blk_hi;
  int max_blocks;
  const int32_t* hblk_lo;
  const int32_t* hblk_hi;
  int max_blocks2;
  void* k_c;            // [B, N_cap, 128]
  void* v_c;
  void* ik_c;           // [B, N_cap, 64]
  int N_cap;
  void* hk_c;           // [B, N2_cap, 128]
  void* hv_c;
  int N2_cap;
  int32_t* idx;         // [B, k]
  int o_dtype;
  void* o;              // [B, H, 128] in o_dtype
  float* lse;           // [B, H]
  void* ho;
  float* hlse;
  int32_t* err;
  // workspace (laid out by the caller)
  int* ctr;             // counters, zeroed by the launch (decode_step_counter_bytes)
  uint32_t* keys;       // [B, N_cap] score keys
  float* part_o;        // [B, na, 64, 128] CSA partials
  float* part_lse;      // [B, na, 64]
  float* hpart_o;       // [B, nh, 64, 128] HCA partials
  float* hpart_lse;     // [B, nh, 64]
  uint32_t* tk_cand;    // [B, 4, 4096] top-k candidate lists
  // plan (decode_step_plan)
  int tps, ns;          // score tiles per item, score items per sequence
  int tpa, na;          // CSA key tiles per share, shares per sequence
  int tph, nh;          // HCA
  int grid;
};
bool decode_step_plan(StepArgs& a, int num_sms);
size_t decode_step_counter_bytes(int B);
cudaError_t launch_decode_step(const StepArgs& a, cudaStream_t st);

// Backward of the attention branches (the key list as in AttnArgs, fixed)
// and of the block pooling; every gradient is added (fp32 atomics) into the
// caller's buffers.
struct AttnBwdArgs {
  int dtype, B, T, H, d;
  float sm_scale;
  const void* q;        // [B*T, H, d]
  const int32_t* q_pos;
  const void* kc;       // [B, N_cap, d]
  const void* vc;
  int N_cap;
  const int32_t* idx;   // [B*T, k] when gather
  int gather, k, m;
  const void* kr;       // [B, R, d]
  const void* vr;
  int R, W;
  const float* o;       // [B*T, H, d] forward output
  const float* lse;     // [B*T, H] forward LSE
  const float* dout;    // [B*T, H, d]
  float* dq;            // [B*T, H, d]
  float* dkc;           // [B, N_cap, d]
  float* dvc;
  float* dkr;           // [B, R, d]
  float* dvr;
  int nsplit, split_tiles;   // key tiles of attend_backward_key_tile() keys
  int32_t* err;
};
cudaError_t launch_attend_backward(const AttnBwdArgs& a, cudaStream_t st);
size_t attend_backward_smem(int H, int d);
int attend_backward_key_tile();

struct CompressBwdArgs {
  int dtype, B, d, m;
  const void* k_raw;    // [B, R, d]
  const void* v_raw;
  const float* z;       // [B, R]
  int R;
  const int32_t* blk_lo;
  const int32_t* blk_hi;
  int max_blocks;
  const float* dkc;     // [B, N_cap, d]
  const float* dvc;
  int N_cap;
  float* dkr;           // [B, R, d]
  float* dvr;
  float* dz;            // [B, R]
  int32_t* err;
};
cudaError_t launch_compress_backward(const CompressBwdArgs& a, cudaStream_t st);

struct MergeArgs {
  int n;
  const float* o_parts[8];
  const float* lse_parts[8];
  int64_t rows;
  int d;
  void* o;
  int o_dtype;
  float* lse;
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t st);

}  // namespace sa
