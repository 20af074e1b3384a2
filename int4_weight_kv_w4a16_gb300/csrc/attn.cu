// Single-query GQA decode attention over the INT4 rotated KV cache.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract: decode reads an INT4 KV-cache copy whose keys follow the
// Tensor Core fragment layout; a block-diagonal Hadamard transform is applied
// to the cache, and (explainer, Hadamard paragraph) correspondingly before and
// after: the query is rotated the same way (in the QKV epilogue) and the
// attention output is rotated back here.
//
// Grid (NC, kv-head, sequence); the NC CTAs of one (sequence, kv-head) form a
// thread-block cluster and split the context into NC contiguous ranges of
// 64-position tiles.  In a CTA:
//   warp 4 (producer) streams the range's tiles (key codes, value codes, key
//     and value scales: four 1-D bulk copies per tile) through a ring of
//     shared-memory stages with mbarrier completion;
//   warps 0..3 (consumers) take one 16-position sub-tile of every tile:
//     S = q' K^T: mma.m16n8k16 f16, A = the G query heads of this kv-head
//       (rows >= G are zero) as an fp16 pair hi + lo of the fp32 query (two
//       MMAs), B = key codes converted in registers (exact);
//     score = S * key_scale * log2(e)/sqrt(d);
//     online softmax in fp32 (running max m, normalizer l, output rescale);
//     O += P V: A = fp16(p * value_scale) as an fp16 pair hi + lo, B = value
//       codes converted in registers.
// The 4 warps merge (m, l, O) in shared memory.  Then the cluster synchronises
// (hardware cluster barrier) and the leader CTA reads the other ranges'
// (m, l, O) from their shared memory (distributed shared memory), merges them
// in range order, divides by l, undoes the rotation (fp32 Hadamard) and
// stores bf16; a second cluster barrier keeps every CTA's shared memory alive
// until the leader is done.  No CTA leaves early, so every thread reaches
// both barriers; the ring waits are bounded.
#include "futr_internal.cuh"
#include "proj.cuh"

namespace futr {

namespace {

constexpr int kAttnCW = 4;                        // consumer warps
constexpr int kAttnThreads = (kAttnCW + 1) * 32;  // + producer warp
constexpr int kTilePos = 16 * kAttnCW;            // positions per ring stage: one 16-position sub-tile per warp
constexpr int kAttnRing = 4;
constexpr int kMaxCluster = 16;

template <int D>
struct AttnLayout {
  static constexpr int kCodes = kTilePos * D / 2;            // key (or value) codes of a tile, bytes
  static constexpr int kStage = 2 * kCodes + 4 * kTilePos;   // + key and value scales (fp16)
  // after the ring: the query A fragments [D/16][hi, lo][32 lanes] (uint4);
  // then floats cm, cl [warps][G]; co [warps][G][D]; mO [G][D]; mm, ml [G];
  // wm, wl [kMaxCluster][G]
  static constexpr int kQFrag = (D / 16) * 2 * 32 * 16;
  __host__ __device__ static int floats(int G) { return 2 * kAttnCW * G + kAttnCW * G * D + G * D + 2 * G + 2 * kMaxCluster * G; }
  __host__ __device__ static size_t bytes(int G) {
    return (size_t)kAttnRing * kStage + kQFrag + 4 * (size_t)floats(G) + 2 * kAttnRing * 8;
  }
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
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

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 3) attn_kernel(const AttnArgs a) {
  constexpr int J = D / 32;
  using Lay = AttnLayout<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int sp = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z, NC = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int G = a.G, cap = a.kv.cap;

  uint8_t* stages = smem;
  uint4* qf = reinterpret_cast<uint4*>(smem + kAttnRing * Lay::kStage);  // [D/16][2][32]
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

  if (tid == 0) {
    for (int i = 0; i < kAttnRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kAttnCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  // pos is an input of the step (the previous kernel does not write it), so the
  // range is known before the wait; the first tiles are pulled into L2 now
  // (a prefetch cannot return stale data: the copies after the wait read
  // through L2, which holds the new token's entries once written)
  const int p = a.pos[b];
  const bool pos_ok = p >= 0 && p < cap;
  const int L = pos_ok ? p + 1 : 0;
  const int T = (L + kTilePos - 1) / kTilePos;
  const int tile0 = (int)((long long)sp * T / NC), ntiles = (int)((long long)(sp + 1) * T / NC) - tile0;
  const uint8_t* strm = a.kv.stream(b, kvh);
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
  pdl_wait();  // q' and the new token's cache entries come from the previous kernel
  bool ok = true;

  if (warp == kAttnCW) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const unsigned long long deadline = global_ns() + kWaitNs;
      auto issue = [&](int slot, int i) {
        const int c0 = (tile0 + i) * kTilePos;
        const int n16 = (min(kTilePos, L - c0) + 15) & ~15;  // c0 + n16 <= round16(L) <= cap
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
      for (int i = 0; i < pre; ++i) issue(i, i);
      int slot = 0;
      uint32_t phase = 0;
      for (int i = kAttnRing; i < ntiles; ++i) {
        if (!mbar_wait_until(&empty[slot], phase, deadline)) {
          set_err(a.err, FUTR_ERR_TIMEOUT);
          break;
        }
        issue(slot, i);
        if (++slot == kAttnRing) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ----------------------------------------------------------- consumers --
    // query fragments (A operand of q.k), once per CTA into shared memory:
    // rows = heads of this group, padded to 16; each fp32 pair becomes an
    // fp16 hi register and an fp16 lo register (the remainder)
    {
      const float* q = a.qrot + ((size_t)b * a.Hq + (size_t)kvh * G) * D;
      const float2 zero = make_float2(0.f, 0.f);
      for (int item = tid; item < (D / 16) * 32; item += kAttnCW * 32) {
        const int ks = item >> 5, ln = item & 31, gq = ln >> 2, tq = ln & 3;
        const int c = 16 * ks + 2 * tq;
        const float2 f0 = gq < G ? *reinterpret_cast<const float2*>(q + gq * D + c) : zero;
        const float2 f1 = gq + 8 < G ? *reinterpret_cast<const float2*>(q + (gq + 8) * D + c) : zero;
        const float2 f2 = gq < G ? *reinterpret_cast<const float2*>(q + gq * D + c + 8) : zero;
        const float2 f3 = gq + 8 < G ? *reinterpret_cast<const float2*>(q + (gq + 8) * D + c + 8) : zero;
        uint4 hi, lo;
        split_half2(f0.x, f0.y, hi.x, lo.x);
        split_half2(f1.x, f1.y, hi.y, lo.y);
        split_half2(f2.x, f2.y, hi.z, lo.z);
        split_half2(f3.x, f3.y, hi.w, lo.w);
        qf[(2 * ks) * 32 + ln] = hi;
        qf[(2 * ks + 1) * 32 + ln] = lo;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kAttnCW * 32) : "memory");  // consumers only
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[D / 8][4];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nd][e] = 0.f;

    const unsigned long long deadline = global_ns() + kWaitNs;
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < ntiles; ++i) {
      if (!mbar_wait_until(&full[slot], phase, deadline)) {
        ok = false;
        break;
      }
      const uint8_t* Ks = stages + (size_t)slot * Lay::kStage;
      const uint8_t* Vs = Ks + Lay::kCodes;
      const __half* ksc = reinterpret_cast<const __half*>(Ks + 2 * Lay::kCodes);
      const __half* vsc = ksc + kTilePos;
      const int npos = min(kTilePos, L - (tile0 + i) * kTilePos);
      if (16 * warp < npos) {
      // S = q' K^T for the two 8-position halves h; the hi and lo query
      // parts accumulate separately (four independent MMA chains)
      float s[2][4], s_lo[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[h][e] = s_lo[h][e] = 0.f;
      const uint32_t* kw0 = reinterpret_cast<const uint32_t*>(Ks + (size_t)(2 * warp) * (4 * D) + lane * (D / 8));
      const uint32_t* kw1 = reinterpret_cast<const uint32_t*>(Ks + (size_t)(2 * warp + 1) * (4 * D) + lane * (D / 8));
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        const uint4 h0 = qf[(4 * j) * 32 + lane], l0q = qf[(4 * j + 1) * 32 + lane];
        const uint4 h1 = qf[(4 * j + 2) * 32 + lane], l1q = qf[(4 * j + 3) * 32 + lane];
        const uint32_t qa0[4] = {h0.x, h0.y, h0.z, h0.w}, ql0[4] = {l0q.x, l0q.y, l0q.z, l0q.w};
        const uint32_t qa1[4] = {h1.x, h1.y, h1.z, h1.w}, ql1[4] = {l1q.x, l1q.y, l1q.z, l1q.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t kk[4];
          nib4_f16x2(h == 0 ? kw0[j] : kw1[j], kk);
          const uint32_t k0 = kk[0], k1 = kk[1], k2 = kk[2], k3 = kk[3];
          mma_f16_16816(s[h], qa0, k0, k1);
          mma_f16_16816(s[h], qa1, k2, k3);
          mma_f16_16816(s_lo[h], ql0, k0, k1);
          mma_f16_16816(s_lo[h], ql1, k2, k3);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[h][e] += s_lo[h][e];
      float sc[2][4], vsv[2][2];
      bool valid[2][2];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pl = 16 * warp + 8 * h + 2 * t + e;
          valid[h][e] = pl < npos;
          const float kscale = valid[h][e] ? __half2float(ksc[pl]) * a.qk_scale_log2 : 0.f;
          vsv[h][e] = valid[h][e] ? __half2float(vsc[pl]) : 0.f;
          sc[h][e] = valid[h][e] ? s[h][e] * kscale : -INFINITY;
          sc[h][2 + e] = valid[h][e] ? s[h][2 + e] * kscale : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float corr0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
      const float corr1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
      float pr[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pr[h][e] = valid[h][e] ? exp2f(sc[h][e] - mn0) : 0.f;
          pr[h][2 + e] = valid[h][e] ? exp2f(sc[h][2 + e] - mn1) : 0.f;
        }
      l0 = l0 * corr0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
      l1 = l1 * corr1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
      m0 = mn0;
      m1 = mn1;
      // rescale O only when some row's running max moved (corr = 1 otherwise:
      // the product would leave O unchanged)
      if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          o[nd][0] *= corr0;
          o[nd][1] *= corr0;
          o[nd][2] *= corr1;
          o[nd][3] *= corr1;
        }
      }
      // P operand = p * value_scale as an fp16 pair hi + lo (hi = fp16(v),
      // lo = fp16(v - hi)): two MMAs keep ~22 bits of each weight.
      uint32_t pa[4], pl[4];
      split_half2(pr[0][0] * vsv[0][0], pr[0][1] * vsv[0][1], pa[0], pl[0]);
      split_half2(pr[0][2] * vsv[0][0], pr[0][3] * vsv[0][1], pa[1], pl[1]);
      split_half2(pr[1][0] * vsv[1][0], pr[1][1] * vsv[1][1], pa[2], pl[2]);
      split_half2(pr[1][2] * vsv[1][0], pr[1][3] * vsv[1][1], pa[3], pl[3]);
      const uint32_t* vw = reinterpret_cast<const uint32_t*>(Vs + (size_t)warp * (8 * D) + lane * (D / 4));
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        uint32_t vv[4];
        nib4_f16x2(vw[j], vv);
        const uint32_t v0 = vv[0], v1 = vv[1], v2 = vv[2], v3 = vv[3];
        mma_f16_16816(o[2 * j], pa, v0, v1);
        mma_f16_16816(o[2 * j + 1], pa, v2, v3);
        mma_f16_16816(o[2 * j], pl, v0, v1);
        mma_f16_16816(o[2 * j + 1], pl, v2, v3);
      }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the stage
      if (++slot == kAttnRing) {
        slot = 0;
        phase ^= 1u;
      }
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // this warp's (m, l, O) rows to shared memory
    if (g < G) {
      if (t == 0) {
        cm[warp * G + g] = m0;
        cl[warp * G + g] = l0;
      }
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        co[(warp * G + g) * D + 8 * nd + 2 * t] = o[nd][0];
        co[(warp * G + g) * D + 8 * nd + 2 * t + 1] = o[nd][1];
      }
    }
    if (g + 8 < G) {
      if (t == 0) {
        cm[warp * G + g + 8] = m1;
        cl[warp * G + g + 8] = l1;
      }
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        co[(warp * G + g + 8) * D + 8 * nd + 2 * t] = o[nd][2];
        co[(warp * G + g + 8) * D + 8 * nd + 2 * t + 1] = o[nd][3];
      }
    }
  }
  if (!ok) set_err(a.err, FUTR_ERR_TIMEOUT);
  __syncthreads();

  // ---- merge the 4 warps: (mO, mm, ml) of this range
  for (int e = tid; e < G * D; e += kAttnThreads) {
    const int r = e / D, i = e % D;
    float M = -INFINITY;
    for (int w = 0; w < kAttnCW; ++w) M = fmaxf(M, cm[w * G + r]);
    float Lr = 0.f, Or = 0.f;
    for (int w = 0; w < kAttnCW; ++w) {
      const float mw = cm[w * G + r];
      const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
      Lr += cl[w * G + r] * wt;
      Or += co[(w * G + r) * D + i] * wt;
    }
    mO[e] = Or;
    if (i == 0) {
      mm[r] = M;
      ml[r] = Lr;
    }
  }
  __syncthreads();
  if (NC > 1) cluster_sync_all();  // every range's (mO, mm, ml) is complete

  if (sp == 0) {
    // ---- the leader merges the NC ranges in range order
    for (int i = tid; i < NC * G; i += kAttnThreads) {
      const int r = i / G, h = i - r * G;
      const float vm = r == 0 ? mm[h] : ld_dsmem(&mm[h], (uint32_t)r);
      const float vl = r == 0 ? ml[h] : ld_dsmem(&ml[h], (uint32_t)r);
      wm[i] = vm;
      wl[i] = vl;
    }
    __syncthreads();
    if (tid < G) {
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
    float4* mO4 = reinterpret_cast<float4*>(mO);
    for (int e4 = tid; e4 < G * D / 4; e4 += kAttnThreads) {
      const int h = (4 * e4) / D;
      // every range's value first (independent remote loads in flight), then
      // the weighted sum in range order
      float4 v[kMaxCluster];
      v[0] = mO4[e4];
#pragma unroll
      for (int r = 1; r < kMaxCluster; ++r)
        if (r < NC) v[r] = ld_dsmem4(&mO4[e4], (uint32_t)r);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < NC) {
          const float wt = wm[r * G + h];
          acc.x += v[r].x * wt; acc.y += v[r].y * wt; acc.z += v[r].z * wt; acc.w += v[r].w * wt;
        }
      mO4[e4] = acc;
    }
    __syncthreads();
    // ---- normalize, rotate back, store bf16 (an empty context stores zeros)
    for (int r = warp; r < G; r += kAttnThreads / 32) {
      const float inv = cm[r] > 0.f ? __fdiv_rn(1.0f, cm[r]) : 0.f;
      float v[J];
#pragma unroll
      for (int j = 0; j < J; ++j) v[j] = mO[r * D + lane + 32 * j] * inv;
      warp_fwht<J>(v, a.nh, a.had_c);
      __nv_bfloat16* out = a.out + ((size_t)b * a.Hq + (size_t)kvh * G + r) * D;
#pragma unroll
      for (int j = 0; j < J; ++j) out[lane + 32 * j] = __float2bfloat16_rn(v[j]);
    }
    if (!pos_ok && kvh == 0 && tid == 0) set_err(a.err, FUTR_ERR_OUT_OF_RANGE);
  }
  if (NC > 1) cluster_sync_all();  // the leader is done reading the other CTAs' shared memory
}

template <int D>
cudaError_t configure_attn(int dev) {
  static unsigned long long configured = 0;  // one bit per device
  if (configured & (1ull << (dev & 63))) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  configured |= 1ull << (dev & 63);
  return cudaSuccess;
}

template <int D>
cudaLaunchConfig_t attn_config(const AttnPlan& p, int Hkv, int batch, cudaStream_t st, cudaLaunchAttribute* attr,
                               bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.NC, (unsigned)Hkv, (unsigned)batch);
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

template <int D>
cudaError_t launch_d(const AttnPlan& p, const AttnArgs& a, cudaStream_t st, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure_attn<D>(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = attn_config<D>(p, a.Hkv, a.batch, st, attr, pdl);
  return cudaLaunchKernelEx(&cfg, attn_kernel<D>, a);
}

// Largest cluster the device schedules for this kernel (at most kMaxCluster).
template <int D>
int max_cluster(size_t smem) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || configure_attn<D>(dev) != cudaSuccess) return 1;
  AttnPlan p{};
  p.NC = 1;
  p.smem = smem;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = attn_config<D>(p, 1, 1, 0, attr, false);
  cfg.numAttrs = 0;  // the query wants no cluster dimension set
  if (cudaOccupancyMaxPotentialClusterSize(&n, attn_kernel<D>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 1;
  }
  return n < kMaxCluster ? n : kMaxCluster;
}

template <int D>
int resident_attn(size_t smem) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || configure_attn<D>(dev) != cudaSuccess) return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<D>, kAttnThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n;
}

}  // namespace

AttnPlan plan_attention(const futr_shape& s, int batch, int cap, int n_sm, int force_split) {
  AttnPlan p{};
  const int G = s.n_q_heads / s.n_kv_heads, D = s.head_dim;
  p.smem = D == 128 ? AttnLayout<128>::bytes(G) : AttnLayout<64>::bytes(G);
  const int lim = D == 128 ? max_cluster<128>(p.smem) : max_cluster<64>(p.smem);
  const int fit = D == 128 ? resident_attn<128>(p.smem) : resident_attn<64>(p.smem);
  // context ranges per (sequence, kv-head): fewest waves of resident CTAs x
  // tiles per range (+ the merge), within the cluster limit and the tiles
  const long long pairs = (long long)batch * s.n_kv_heads, slots = (long long)n_sm * (fit > 0 ? fit : 1);
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
  p.part_floats = 0;
  return p;
}

cudaError_t launch_attention(const AttnPlan& p, AttnArgs a, int d, cudaStream_t st, bool pdl) {
  return d == 128 ? launch_d<128>(p, a, st, pdl) : launch_d<64>(p, a, st, pdl);
}

}  // namespace futr
