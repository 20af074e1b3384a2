// Single-query GQA decode attention over the INT4 rotated KV cache.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract: decode reads an INT4 KV-cache copy whose keys follow the
// Tensor Core fragment layout; a block-diagonal Hadamard transform is applied
// to the cache, and (explainer, Hadamard paragraph) correspondingly before and
// after: the query is rotated the same way (in the QKV epilogue) and the
// attention output is rotated back here.
//
// Grid (NC, kv-head x head sub-group, sequence); the NC CTAs of one
// (sequence, kv-head, sub-group) form a thread-block cluster and split the
// context into NC contiguous ranges of 64-position tiles.  A kv-head's G query
// heads go to ceil(G / 8) sub-groups of at most 8 heads (one for Llama's G of
// 4 and 8).  In a CTA:
//   warp 4 (producer) streams the range's tiles (key codes, value codes, key
//     and value scales: four 1-D bulk copies per tile) through a ring of
//     shared-memory stages with mbarrier completion;
//   warps 0..3 (consumers) take one 16-position sub-tile of every tile and
//     work in the transposed orientation, positions along the MMA's 16 rows:
//     S^T = K q'^T: mma.m16n8k16 f16, A = key codes converted in registers
//       (exact), B = the query heads as columns, each fp32 query as an fp16
//       pair hi + lo: the hi parts take the first half of the columns, the lo
//       parts the second half, so one MMA carries both (4 heads per n-tile of
//       8 columns; 8 heads in two n-tiles);
//     score = (hi + lo column sum) * key_scale * log2(e)/sqrt(d);
//     online softmax in fp32 (running max m, normalizer l, output rescale);
//     O^T += V^T P^T: A = value codes converted in registers, B = fp16(p *
//       value_scale) as an fp16 pair hi + lo in the same column split (the
//       score fragment becomes the B operand by an 8x8 register transpose).
// The 4 warps merge (m, l, O) in shared memory.  Then the cluster synchronises
// (hardware cluster barrier) and the leader CTA reads the other ranges'
// (m, l, O) from their shared memory (distributed shared memory), merges them
// in range order, divides by l, undoes the rotation (fp32 Hadamard) and
// stores bf16; a second cluster barrier keeps every CTA's shared memory alive
// until the leader is done.  No CTA leaves early, so every thread reaches
// both barriers; the ring waits are bounded.
//
// By default the QKV projection leaves its split-K records
// (AttnArgs::qkv_part) and the head epilogue runs here, after the wait: every CTA adds the records
// of its query heads, applies the RMSNorm factor, RoPE and the rotation and
// builds the query fragments from shared memory; in the CTA of the last range
// the producer warp forms the new token's INT4 key and value, and the consumer
// warp whose sub-tile holds that position patches them into its ring stage
// (the copy of that slot predates them) and writes them into the cache.
#include "futr_internal.cuh"
#include "proj.cuh"
#include "attn_dev.cuh"

namespace futr {

namespace {

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The closing barrier publishes nothing: every value the leader read from the
// other CTAs' shared memory has been consumed by its stores before it, so the
// arrival needs no release.
__device__ __forceinline__ void cluster_sync_exit() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(dsmem_addr(local, rank)) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_dsmem4(const float4* local, uint32_t rank) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(dsmem_addr(local, rank))
               : "memory");
  return v;
}

// ------------------------------------------ QKV head epilogue (deferred) --
// The QKV projection left its split records (kEpiQkvRec).  Head task i of
// this CTA: query head hq0 + i for i < Gv, then (kv) the key and the value
// head of kv-head kvh.  qs[i * D + r] = the sum over the splits (in split
// order) of row r of task i's head, batch row b; *ss = the sum of squares of
// x.  All threads of the CTA; loads of 8 splits in flight per item.
template <int D>
__device__ __forceinline__ void sum_qkv_records(const AttnArgs& a, int b, int hq0, int Gv, int kvh, bool kv,
                                                float* qs, float* ss) {
  constexpr int C = D / 4;  // float4 columns of a head
  const int hpr = kRowsPerBlock / D, nt = Gv + (kv ? 2 : 0), S = a.qkv_S;
  const size_t step = (size_t)a.qkv_rec_floats / 4;
  for (int e = threadIdx.x; e < nt * C + 1; e += kAttnThreads) {
    int rb = hq0 / hpr, col = kRecCols - 1;  // the last item: (sum of squares, 0, 0, 0)
    if (e < nt * C) {
      const int i = e / C, c = e - i * C;
      const int hg = i < Gv ? hq0 + i : (i == Gv ? a.Hq + kvh : a.Hq + a.Hkv + kvh);
      rb = hg / hpr;
      col = (hg - rb * hpr) * C + c;
    }
    // debug build: the records read lie inside the region
    if (!FUTR_DCHECK(((size_t)rb * a.qkv_stride + S) * a.qkv_rec_floats <= a.qkv_part_cap &&
                         (size_t)(b + 1) * kRecLd <= (size_t)a.qkv_rec_floats,
                     a.err))
      continue;
    const float4* src = reinterpret_cast<const float4*>(a.qkv_part + (size_t)rb * a.qkv_stride * a.qkv_rec_floats +
                                                        (size_t)b * kRecLd) + col;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < S) v[j] = __ldcg(src + (size_t)(s0 + j) * step);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < S) {
          acc.x += v[j].x; acc.y += v[j].y; acc.z += v[j].z; acc.w += v[j].w;
        }
    }
    if (e < nt * C)
      reinterpret_cast<float4*>(qs)[e] = acc;
    else
      *ss = acc.x;
  }
}

// One head task (one warp): v[j] = element lane + 32 j of the head's sums
// times the RMSNorm factor rn, RoPE (rotate-half, dims i and i + D/2: element
// j pairs j + J/2; cs[j] holds (cos, sin) of dims lane + 32 j) for query and
// key heads, then the fp32 rotation.
template <int D>
__device__ __forceinline__ void head_from_sums(float (&v)[D / 32], const float* sums, float rn, bool rope,
                                               const float2 (&cs)[2], const AttnArgs& a) {
  constexpr int J = D / 32;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < J; ++j) v[j] = sums[lane + 32 * j] * rn;
  if (rope) {
#pragma unroll
    for (int j = 0; j < J / 2; ++j) {
      const float x1 = v[j], x2 = v[j + J / 2];
      v[j] = x1 * cs[j].x - x2 * cs[j].y;
      v[j + J / 2] = x2 * cs[j].x + x1 * cs[j].y;
    }
  }
  warp_fwht<J>(v, a.nh, a.had_c);
}

// The new token (position p, offset r = p - c0 in the tile at c0) into a ring
// stage that holds its tile (one warp): key codes, value nibbles and both
// scales, from tok[0] / tok[1] (int8 codes, dim order) and toks.
template <int D>
__device__ __forceinline__ void patch_new_token(uint8_t* st, int r, int p, const int8_t (*tok)[D],
                                                const __half* toks) {
  using Lay = AttnLayout<D>;
  const int lane = threadIdx.x & 31;
  uint32_t* kw = reinterpret_cast<uint32_t*>(st + (size_t)r * (D / 2));
  if (lane < D / 8) kw[lane] = k_token_word<D>(tok[0], lane);
  uint32_t* vt = reinterpret_cast<uint32_t*>(st + Lay::kCodes + (size_t)(r >> 4) * (8 * D));
  for (int w = lane; w < 8 * (D / 16); w += 32) {
    const VWord vw = v_token_word<D>(tok[1], p, w);
    vt[vw.off] = (vt[vw.off] & ~vw.mask) | vw.bits;
  }
  if (lane == 0) {
    __half* ksc = reinterpret_cast<__half*>(st + 2 * Lay::kCodes);
    ksc[r] = toks[0];
    ksc[kTilePos + r] = toks[1];
  }
  __syncwarp();
}

// NTQ: n-tiles of query columns (1: at most 4 heads, 2: at most 8).
template <int D, int NTQ>
__global__ void __launch_bounds__(kAttnThreads, NTQ == 1 ? 4 : 3) attn_kernel(const AttnArgs a) {
  constexpr int J = D / 32;
  using Lay = AttnLayout<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int nsub = attn_nsub(a.G);
  const int sp = blockIdx.x, kvh = blockIdx.y / nsub, sub = blockIdx.y - kvh * nsub, b = blockIdx.z, NC = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cap = a.kv.cap;
  // G: heads per sub-group (the shared-memory layout); Gv: this sub-group's
  // heads, query heads hq0 .. hq0 + Gv - 1
  const int G = attn_gc(a.G), hq0 = kvh * a.G + sub * G, Gv = min(G, a.G - sub * G);

  uint8_t* stages = smem;
  uint2* qf = reinterpret_cast<uint2*>(smem + kAttnRing * Lay::kStage);  // [D/16][NTQ][32]
  float* cm = reinterpret_cast<float*>(smem + kAttnRing * Lay::kStage + Lay::kQFrag);  // [warps][G]
  float* cl = cm + kAttnCW * G;                                          // [warps][G]
  float* co = cl + kAttnCW * G;                                          // [warps][G][D]
  float* mO = co + kAttnCW * G * D;                                      // [G][D] (16-byte aligned)
  float* mm = mO + G * D;                                                // [G]
  float* ml = mm + G;                                                    // [G]
  float* wm = ml + G;                                                    // [kMaxCluster][G]
  float* wl = wm + kMaxCluster * G;                                      // [kMaxCluster][G]
  uint64_t* full = reinterpret_cast<uint64_t*>(wl + kMaxCluster * G);
  uint64_t* empty = full + kAttnRing;

  // ring stages the producer issued, and whether some wait of this CTA ran out
  // (then the CTA lets the issued copies land before it exits)
  __shared__ int s_issued, s_timeout;
  // deferred QKV epilogue: the head tasks' sums (then q'), the sum of squares
  // of x, the new token's codes and scales and their arrival
  __shared__ __align__(16) float s_qs[(4 * NTQ + 2) * D];
  __shared__ float s_ss;
  __shared__ int8_t s_tok[2][D];
  __shared__ __half s_toks[2];
  __shared__ __align__(8) uint64_t s_kvready;
  if (tid == 0) {
    for (int i = 0; i < kAttnRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kAttnCW);
    }
    mbar_init(&s_kvready, 1);
    fence_mbar_init();
    s_issued = 0;
    s_timeout = 0;
  }
  __syncthreads();
  // the next kernel may launch now; with the QKV records, only once they are
  // summed (its CTAs' weight prefetch would compete with these L2 loads)
  if (a.qkv_part == nullptr) pdl_trigger();
  // pos is an input of the step (the previous kernel does not write it), so the
  // range is known before the wait; the first tiles are pulled into L2 now
  // (a prefetch cannot return stale data: the copies after the wait read
  // through L2, which holds the new token's entries once written)
  const int p = a.pos[b];
  const bool pos_ok = p >= 0 && p < cap;
  const int L = pos_ok ? p + 1 : 0;
  const int T = (L + kTilePos - 1) / kTilePos;
  const int tile0 = (int)((long long)sp * T / NC), ntiles = (int)((long long)(sp + 1) * T / NC) - tile0;
  uint8_t* strm = a.kv.stream(b, kvh);
  if (warp == kAttnCW && lane == 0) {
    for (int i = 0; i < ntiles && i < kAttnRing; ++i) {
      const int c0 = (tile0 + i) * kTilePos;
      const int n16 = (min(kTilePos, L - c0) + 15) & ~15;
      const uint32_t cb = (uint32_t)n16 * (D / 2), sb = (uint32_t)n16 * 2;
      l2_prefetch(strm + (size_t)c0 * (D / 2), cb);
      l2_prefetch(strm + (size_t)cap * (D / 2) + (size_t)c0 * (D / 2), cb);
      l2_prefetch(strm + (size_t)cap * D + 2 * (size_t)c0, sb);
      l2_prefetch(strm + (size_t)cap * D + 2 * (size_t)cap + 2 * (size_t)c0, sb);
    }
  }
  // with the QKV records (deferred head epilogue): the RoPE factors of
  // dims lane + 32 j at position p, loaded now (pos and the table are inputs
  // of the step); the CTA of the last range, which holds position p, also
  // forms the new token's key and value
  const bool defer = a.qkv_part != nullptr;
  const bool kv_task = defer && pos_ok && sp == NC - 1;
  float2 rcs[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
  if (defer) {
    const int half = D / 2, pp = pos_ok ? p : 0;
    rcs[0] = a.rope[(size_t)pp * half + lane];
    if (half > 32) rcs[1] = a.rope[(size_t)pp * half + lane + 32];
  }
  pdl_wait();  // q' (or the QKV records) and the new token's cache entries come from the previous kernel
  bool ok = true;
  const unsigned long long deadline = global_ns() + kWaitNs;
  auto issue = [&](int slot, int i) {
    const int c0 = (tile0 + i) * kTilePos;
    const int n16 = (min(kTilePos, L - c0) + 15) & ~15;  // c0 + n16 <= round16(L) <= cap
    if (!FUTR_DCHECK(c0 >= 0 && c0 + n16 <= cap, a.err)) return;  // debug build
    const uint32_t cb = (uint32_t)n16 * (D / 2), sb = (uint32_t)n16 * 2;
    uint8_t* st = stages + (size_t)slot * Lay::kStage;
    mbar_arrive_expect_tx(&full[slot], 2 * cb + 2 * sb);
    bulk_g2s(st, strm + (size_t)c0 * (D / 2), cb, &full[slot]);
    bulk_g2s(st + Lay::kCodes, strm + (size_t)cap * (D / 2) + (size_t)c0 * (D / 2), cb, &full[slot]);
    bulk_g2s(st + 2 * Lay::kCodes, strm + (size_t)cap * D + 2 * (size_t)c0, sb, &full[slot]);
    bulk_g2s(st + 2 * Lay::kCodes + 2 * kTilePos, strm + (size_t)cap * D + 2 * (size_t)cap + 2 * (size_t)c0, sb,
             &full[slot]);
  };
  const int pre = ntiles < kAttnRing ? ntiles : kAttnRing;
  if (warp == kAttnCW && lane == 0)
    for (int i = 0; i < pre; ++i) issue(i, i);
  float rn = 0.f;
  if (defer) {
    // every thread: the head tasks' sums (the first tiles are landing meanwhile)
    sum_qkv_records<D>(a, b, hq0, Gv, kvh, kv_task, s_qs, &s_ss);
    __syncthreads();
    pdl_trigger();
    rn = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(s_ss, (float)a.hidden) + a.eps));
  }

  if (warp == kAttnCW) {
    // ---------------------------------------------------------- producer --
    if (kv_task) {
      // the new token's key (RoPE, rotation) and value (rotation), INT4 with
      // an fp16 scale each, for the consumer warp whose sub-tile holds it
      float v[J];
      int code[J];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        head_from_sums<D>(v, s_qs + (Gv + t) * D, rn, t == 0, rcs, a);
        const __half sc = warp_quant<J>(v, code);
#pragma unroll
        for (int j = 0; j < J; ++j) s_tok[t][lane + 32 * j] = (int8_t)code[j];
        if (lane == 0) s_toks[t] = sc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_kvready);
    }
    if (lane == 0) {
      int slot = 0, issued = pre;
      uint32_t phase = 0;
      for (int i = kAttnRing; i < ntiles; ++i) {
        if (!mbar_wait_until(&empty[slot], phase, deadline, a.err)) {
          ok = false;
          break;
        }
        issue(slot, i);
        issued = i + 1;
        if (++slot == kAttnRing) {
          slot = 0;
          phase ^= 1u;
        }
      }
      s_issued = issued;
    }
  } else {
    // ----------------------------------------------------------- consumers --
    // query fragments (B operand of K q'^T), once per CTA into shared memory
    if (defer) {
      // the query heads' epilogue: q' in place of the sums; the first range
      // also writes it to qrot
      for (int i = warp; i < Gv; i += kAttnCW) {
        float v[J];
        head_from_sums<D>(v, s_qs + i * D, rn, true, rcs, a);
        float* q = a.qrot + ((size_t)b * a.Hq + hq0 + i) * D;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          s_qs[i * D + lane + 32 * j] = v[j];
          if (sp == 0) q[lane + 32 * j] = v[j];
        }
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kAttnCW * 32) : "memory");  // consumers only
      build_qfrag<D, NTQ, true>(s_qs, Gv, qf, tid, kAttnCW * 32);
    } else {
      build_qfrag<D, NTQ>(a.qrot + ((size_t)b * a.Hq + hq0) * D, Gv, qf, tid, kAttnCW * 32);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kAttnCW * 32) : "memory");  // consumers only
    AttnWarp<D, NTQ> aw;
    aw.init();
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < ntiles; ++i) {
      if (!mbar_wait_until(&full[slot], phase, deadline, a.err)) {
        ok = false;
        break;
      }
      const int c0 = (tile0 + i) * kTilePos;
      if (kv_task && i == ntiles - 1 && warp == ((p - c0) >> 4)) {
        // this warp's sub-tile holds the new token: its cache slot held no
        // entry of this step when the tile was copied, so it is patched in
        // the stage, then written to the cache for the later steps
        if (!mbar_wait_until(&s_kvready, 0, deadline, a.err)) {
          ok = false;
          break;
        }
        patch_new_token<D>(stages + (size_t)slot * Lay::kStage, p - c0, p, s_tok, s_toks);
        put_k_token<D>(strm, cap, p, s_tok[0], s_toks[0]);
        put_v_token<D>(strm, cap, p, s_tok[1], s_toks[1]);
      }
      aw.tile(stages + (size_t)slot * Lay::kStage, min(kTilePos, L - (tile0 + i) * kTilePos), qf, a.qk_scale_log2);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the stage
      if (++slot == kAttnRing) {
        slot = 0;
        phase ^= 1u;
      }
    }
    aw.finish(cm, cl, co, G, Gv);
  }
  if (!ok) {
    record_timeout(a.err);
    s_timeout = 1;
  }
  __syncthreads();

  // ---- merge the 4 warps: (mO, mm, ml) of this range
  merge_warps(cm, cl, co, mO, mm, ml, wm, G, Gv, D, tid, kAttnThreads, []() { __syncthreads(); });
  __syncthreads();
  if (NC > 1) cluster_sync_all();  // every range's (mO, mm, ml) is complete

  if (sp == 0) {
    // ---- the leader merges the NC ranges in range order
    float4* mO4 = reinterpret_cast<float4*>(mO);
    // With at most one float4 of O per thread (up to 4 heads of 128 dims),
    // its NC range values are loaded together with the ranges' (m, l), before
    // the weights are known: one round of remote loads instead of two.
    const int n4 = Gv * D / 4;
    const bool one = n4 <= kAttnThreads;
    float4 v[kMaxCluster];
    if (one && tid < n4) {
      v[0] = mO4[tid];
#pragma unroll
      for (int r = 1; r < kMaxCluster; ++r)
        if (r < NC) v[r] = ld_dsmem4(&mO4[tid], (uint32_t)r);
    }
    for (int i = tid; i < NC * G; i += kAttnThreads) {
      const int r = i / G, h = i - r * G;
      if (h >= Gv) continue;
      const float vm = r == 0 ? mm[h] : ld_dsmem(&mm[h], (uint32_t)r);
      const float vl = r == 0 ? ml[h] : ld_dsmem(&ml[h], (uint32_t)r);
      wm[i] = vm;
      wl[i] = vl;
    }
    __syncthreads();
    if (tid < Gv) {
      float M = -INFINITY;
      for (int r = 0; r < NC; ++r) M = fmaxf(M, wm[r * G + tid]);
      float Lr = 0.f;
      for (int r = 0; r < NC; ++r) {
        const float wt = wm[r * G + tid] == -INFINITY ? 0.f : exp2f(wm[r * G + tid] - M);
        wm[r * G + tid] = wt;
        Lr += wl[r * G + tid] * wt;
      }
      cm[tid] = Lr;  // total normalizer of head row tid
    }
    __syncthreads();
    if (one) {
      if (tid < n4) {
        const int h = (4 * tid) / D;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < NC) {
            const float wt = wm[r * G + h];
            acc.x += v[r].x * wt; acc.y += v[r].y * wt; acc.z += v[r].z * wt; acc.w += v[r].w * wt;
          }
        mO4[tid] = acc;  // only this thread reads or writes this float4
      }
    } else {
      for (int e4 = tid; e4 < n4; e4 += kAttnThreads) {
        const int h = (4 * e4) / D;
        // every range's value first (independent remote loads in flight), then
        // the weighted sum in range order
        float4 w[kMaxCluster];
        w[0] = mO4[e4];
#pragma unroll
        for (int r = 1; r < kMaxCluster; ++r)
          if (r < NC) w[r] = ld_dsmem4(&mO4[e4], (uint32_t)r);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < NC) {
            const float wt = wm[r * G + h];
            acc.x += w[r].x * wt; acc.y += w[r].y * wt; acc.z += w[r].z * wt; acc.w += w[r].w * wt;
          }
        mO4[e4] = acc;
      }
    }
    __syncthreads();
    // ---- normalize, rotate back, store bf16 (an empty context stores zeros)
    for (int r = warp; r < Gv; r += kAttnThreads / 32) {
      const float inv = cm[r] > 0.f ? __fdiv_rn(1.0f, cm[r]) : 0.f;
      float v[J];
#pragma unroll
      for (int j = 0; j < J; ++j) v[j] = mO[r * D + lane + 32 * j] * inv;
      warp_fwht<J>(v, a.nh, a.had_c);
      __nv_bfloat16* out = a.out + ((size_t)b * a.Hq + (size_t)hq0 + r) * D;
#pragma unroll
      for (int j = 0; j < J; ++j) out[lane + 32 * j] = __float2bfloat16_rn(v[j]);
    }
    if (!pos_ok && kvh == 0 && tid == 0) set_err(a.err, FUTR_ERR_OUT_OF_RANGE);
  }
  if (NC > 1) cluster_sync_exit();  // the leader is done reading the other CTAs' shared memory
  if (s_timeout && tid == 0) drain_ring(full, kAttnRing, s_issued);
}

template <int D, int NTQ>
cudaError_t configure_attn(int dev) {
  static DeviceOnce configured;
  if (configured.done(dev)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, NTQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<D, NTQ>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<D, NTQ>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  configured.mark(dev);
  return cudaSuccess;
}

cudaLaunchConfig_t attn_config(const AttnPlan& p, int ny, int batch, cudaStream_t st, cudaLaunchAttribute* attr,
                               bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.NC, (unsigned)ny, (unsigned)batch);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = (unsigned)p.NC;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

template <int D, int NTQ>
cudaError_t launch_d(const AttnPlan& p, const AttnArgs& a, cudaStream_t st, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure_attn<D, NTQ>(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = attn_config(p, a.Hkv * attn_nsub(a.G), a.batch, st, attr, pdl);
  return cudaLaunchKernelEx(&cfg, attn_kernel<D, NTQ>, a);
}

// Largest cluster the device schedules for this kernel (at most kMaxCluster).
template <int D, int NTQ>
int max_cluster(size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || configure_attn<D, NTQ>(dev) != cudaSuccess) return 1;
  return remembered(occ_key(dev, D, NTQ, smem), [&]() {
    int n = 0;
    AttnPlan p{};
    p.NC = 1;
    p.smem = smem;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = attn_config(p, 1, 1, 0, attr, false);
    cfg.numAttrs = 0;  // the query wants no cluster dimension set
    if (cudaOccupancyMaxPotentialClusterSize(&n, attn_kernel<D, NTQ>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      return 1;
    }
    return n < kMaxCluster ? n : kMaxCluster;
  });
}

template <int D, int NTQ>
int resident_attn(size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || configure_attn<D, NTQ>(dev) != cudaSuccess) return 1;
  return remembered(occ_key(dev, D, NTQ, smem), [&]() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<D, NTQ>, kAttnThreads, smem) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    return n;
  });
}

// The four instantiations, by head dim and query n-tiles.
int max_cluster_any(int D, int ntq, size_t smem) {
  if (D == 128) return ntq == 1 ? max_cluster<128, 1>(smem) : max_cluster<128, 2>(smem);
  return ntq == 1 ? max_cluster<64, 1>(smem) : max_cluster<64, 2>(smem);
}

int resident_attn_any(int D, int ntq, size_t smem) {
  if (D == 128) return ntq == 1 ? resident_attn<128, 1>(smem) : resident_attn<128, 2>(smem);
  return ntq == 1 ? resident_attn<64, 1>(smem) : resident_attn<64, 2>(smem);
}

}  // namespace

AttnPlan plan_attention(const futr_shape& s, int batch, int cap, int n_sm, int force_split) {
  AttnPlan p{};
  const int G = s.n_q_heads / s.n_kv_heads, D = s.head_dim, gc = attn_gc(G), ntq = gc <= 4 ? 1 : 2;
  p.smem = D == 128 ? AttnLayout<128>::bytes(gc) : AttnLayout<64>::bytes(gc);
  const int lim = max_cluster_any(D, ntq, p.smem);
  const int fit = resident_attn_any(D, ntq, p.smem);
  // context ranges per (sequence, kv-head, head sub-group): fewest waves of
  // resident CTAs x tiles per range (+ the merge), within the cluster limit
  // and the tiles
  // (85 % of the resident slots: with programmatic launch the previous
  // kernel's last CTAs still hold part of the SMs when these start, so a
  // grid that exactly fills the slots runs as two waves)
  const long long pairs = (long long)batch * s.n_kv_heads * attn_nsub(G);
  const long long slots = (long long)(0.85 * n_sm * (fit > 0 ? fit : 1));
  const int tiles = (cap + kTilePos - 1) / kTilePos;
  int nc = 1;
  double best = 1e30;
  for (int c = 1; c <= lim && c <= tiles; ++c) {
    const long long waves = (pairs * c + slots - 1) / slots;
    const double cost = (double)waves * ((tiles + c - 1) / c + 2) + (c > 1 ? 1.0 : 0.0);
    if (cost < best - 1e-9) {
      best = cost;
      nc = c;
    }
  }
  if (force_split > 0) nc = force_split < lim ? force_split : lim;
  if (nc > tiles) nc = tiles;
  if (nc < 1) nc = 1;
  p.NC = nc;
  p.one_sub = attn_nsub(G) == 1;
  p.part_floats = 0;
  return p;
}

cudaError_t launch_attention(const AttnPlan& p, AttnArgs a, int d, cudaStream_t st, bool pdl) {
  const bool one = attn_gc(a.G) <= 4;
  if (d == 128) return one ? launch_d<128, 1>(p, a, st, pdl) : launch_d<128, 2>(p, a, st, pdl);
  return one ? launch_d<64, 1>(p, a, st, pdl) : launch_d<64, 2>(p, a, st, pdl);
}

}  // namespace futr
