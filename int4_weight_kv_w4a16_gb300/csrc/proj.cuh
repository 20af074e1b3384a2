// Arguments and launch plans of the W4A16 projection and attention kernels.
#pragma once

#include <cuda.h>

#include "futr_internal.cuh"

namespace futr {

constexpr int kMaxRing = 8;         // bulk-copy ring depth (stages)
constexpr int kTileLd = 136;        // bf16 row of an activation tile in shared memory (128 + pad)
constexpr int kRedLd = 132;         // fp32 row of the epilogue tile (bank-conflict padding)
constexpr int kRecCols = kRowsPerBlock / 4 + 1;  // float4 columns per batch row of a split record
constexpr int kRecLd = 4 * kRecCols;             // floats per batch row of a split record
constexpr int kProjMaxSmem = 200 * 1024;

constexpr int kEpiResid = 0;
constexpr int kEpiSwiglu = 1;
constexpr int kEpiQkv = 2;
// QKV whose CTAs only write their split records (with the sums of squares)
// and leave: the attention kernel adds them and runs the head epilogue
constexpr int kEpiQkvRec = 3;

struct ProjArgs {
  const uint8_t* w;              // section base of the packed blob
  const __nv_bfloat16* xin;      // activations [batch][K]
  int K, n_groups, S, batch;
  int part_stride;               // records per row block in `part` (S in the one-projection kernels)
  int ring, stage_bytes, off_misc, rec_floats;
  float* part;                   // split-K partial records [n_rb][S][rec_floats]
  unsigned* cnt;                 // arrival counters [n_rb]
  int* err;
  float eps;
  int cluster;                   // the S CTAs of a row block form a cluster (reduction in shared memory)
  // extents the debug build checks accesses against: floats of `part`, rows
  // blocks of the section, elements of `out` (RESID / SWIGLU)
  size_t part_cap, out_cap;
  int n_rb;
  // failure injection for tests: when 1, CTA 0 issues no copy at all, so its
  // consumers' bounded waits run out (0 in every normal call)
  int withhold;
  // RESID / SWIGLU output
  const __nv_bfloat16* resid;    // RESID: [batch][out_ld]
  __nv_bfloat16* out;
  int out_ld;
  // QKV
  const uint64_t* blob_magic;
  float* qrot;                   // [batch][Hq][d] rotated query, fp32
  KvView kv;
  const int* pos;
  const float2* rope;            // [cap][d/2]
  int Hq, Hkv, d, nh;
  float had_c;
};

struct ProjPlan {
  int n_rb, n_groups, nt, S, epi;
  int s_cap;                     // largest split any plan of this shape and batch can choose
  bool tc;                       // tensor-core kernel (batch 17..32)
  bool cluster;                  // mma.sync kernel with the split-K reduction inside a cluster of S CTAs
  int ring, stage_bytes, off_misc, rec_floats;
  size_t smem;
  size_t part_floats;            // split records of this plan
  size_t part_cap_floats;        // split records at s_cap (what a workspace reserves)
};

ProjPlan plan_projection(int rows, int cols, int batch, int n_sm, int force_split, int epi);
cudaError_t launch_projection(int epi, const ProjPlan& p, ProjArgs a, cudaStream_t st, bool pdl);

struct AttnArgs {
  float* qrot;                   // [batch][Hq][d] rotated query, fp32 (written here with qkv_part)
  KvView kv;
  const int* pos;
  int batch, Hq, Hkv, G, nh;
  float qk_scale_log2;           // log2(e) / sqrt(d)
  float had_c;
  __nv_bfloat16* out;            // [batch][Hq*d]
  int* err;
  // The QKV projection's split records when it left its head epilogue to this
  // kernel (kEpiQkvRec), else null: [row block][qkv_S][qkv_rec_floats]
  // (row block stride qkv_stride records).  The CTAs then add the records of
  // their query heads (and, in the CTA whose range holds the new position,
  // of their kv-head's key and value rows), apply the RMSNorm factor, RoPE
  // and the rotation, write q' to qrot (first range) and the new token's
  // codes into the cache (last range).
  const float* qkv_part;
  int qkv_S, qkv_stride, qkv_rec_floats;
  size_t qkv_part_cap;           // floats of qkv_part (debug-build bounds checks)
  int hidden;                    // inputs of the QKV projection (RMSNorm mean)
  float eps;
  const float2* rope;            // [cap][d/2]
};

struct AttnPlan {
  int NC;                        // context ranges (cluster size) per (sequence, kv-head)
  bool one_sub;                  // one head sub-group (one cluster) per kv-head and sequence
  size_t smem;
  size_t part_floats;            // global scratch (none: ranges merge in distributed shared memory)
};

// Tensor map of a tensor-core projection's activation tiles (defined with the
// other tensor maps in step.cu).
bool make_act_tile_map(CUtensorMap* m, const void* x, int rows, int K);
bool make_proj_tile_map(CUtensorMap* m, const void* x, int rows, int K, int box_rows);

AttnPlan plan_attention(const futr_shape& s, int batch, int cap, int n_sm, int force_split);
cudaError_t launch_attention(const AttnPlan& p, AttnArgs a, int d, cudaStream_t st, bool pdl);

// ------------------------------------------ persistent whole-block kernel --
constexpr int kBlockMaxBatch = 16;       // batch tiles 1..2 of mma.sync
constexpr int kBlockMaxSmem = 200 * 1024;  // dynamic shared memory limit asked for (static use comes on top)

// One projection phase of the block kernel: its section, row blocks, input
// groups and the CTAs that take part (each a contiguous range of units).
struct BlockPhase {
  const uint8_t* w;
  int n_rb, n_groups, ne;
};

struct BlockArgs {
  ProjArgs pa[4];                // epilogue arguments of QKV, O, gate/up, down
  BlockPhase ph[4];
  AttnArgs at;                   // attention (qrot, cache, pos, out = o, ...)
  int n_ctx, NC, nsub, gc, arec_floats;  // contexts = sequence x kv-head x sub-group of gc query heads
  float* apart;                  // context-range records [n_ctx][NC][arec_floats]
  unsigned* actx;                // arrival counters [n_ctx] (self-resetting)
  unsigned* done;                // [6]: completed row blocks / contexts per phase, CTAs that left
  int ring, stage_bytes, off_scratch, off_misc;
  int* err;
};

struct BlockPlan {
  bool ok;
  int nt, ntq, nsub, gc, stage_bytes, ring, off_scratch, off_misc;
  int grid;                      // CTAs of the launch (all resident)
  int grid_cap;                  // the most any plan of this shape uses (workspace bound)
  int n_ctx, NC, arec_floats;
  size_t smem;
};

// fixed_ctas_per_sm: 0 = the default (two per SM, fewer if the occupancy
// answer is lower).
BlockPlan plan_block(const futr_shape& s, int batch, int cap, int n_sm, int fixed_ctas_per_sm);
cudaError_t launch_block(const BlockPlan& p, const BlockArgs& a, const CUtensorMap* maps, cudaStream_t st, bool pdl);

}  // namespace futr
