// Device code of the INT4 decode attention shared by the one-step attention
// kernel (attn.cu) and the persistent whole-block kernel (block.cu): the
// ring-stage layout of a 64-position tile, the query fragments, one consumer
// warp's work on a tile (scores, online softmax, P V) and the merge of the
// consumer warps' partial results.
#pragma once

#include "futr_internal.cuh"
#include "proj.cuh"

namespace futr {
namespace {

constexpr int kAttnCW = 4;                        // consumer warps
constexpr int kAttnThreads = (kAttnCW + 1) * 32;  // + producer warp
constexpr int kTilePos = 16 * kAttnCW;            // positions per ring stage: one 16-position sub-tile per warp
constexpr int kAttnRing = 4;
constexpr int kMaxCluster = 16;

constexpr int kMaxSubHeads = 8;  // query heads of one CTA (two n-tiles of hi + lo columns)

// Query heads of one sub-group, and the sub-groups of a kv-head.
__host__ __device__ inline int attn_nsub(int G) { return (G + kMaxSubHeads - 1) / kMaxSubHeads; }
__host__ __device__ inline int attn_gc(int G) { return (G + attn_nsub(G) - 1) / attn_nsub(G); }

template <int D>
struct AttnLayout {
  static constexpr int kCodes = kTilePos * D / 2;            // key (or value) codes of a tile, bytes
  static constexpr int kStage = 2 * kCodes + 4 * kTilePos;   // + key and value scales (fp16)
  // after the ring: the query B fragments [D/16][2 n-tiles][32 lanes] (uint2);
  // then floats cm, cl [warps][G]; co [warps][G][D]; mO [G][D]; mm, ml [G];
  // wm, wl [kMaxCluster][G] (G = the heads of one sub-group)
  static constexpr int kQFrag = (D / 16) * 2 * 32 * 8;
  __host__ __device__ static int floats(int G) { return 2 * kAttnCW * G + kAttnCW * G * D + G * D + 2 * G + 2 * kMaxCluster * G; }
  __host__ __device__ static size_t bytes(int G) {
    return (size_t)kAttnRing * kStage + kQFrag + 4 * (size_t)floats(G) + 2 * kAttnRing * 8;
  }
};

// 2^x by the hardware approximation (relative error ~2^-22; arguments here are
// <= 0, results below 2^-126 flush to zero, 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The B fragments of K q'^T for one head sub-group, once per context into
// shared memory qf[(ks * NTQ + nt) * 32 + lane]: column c of n-tile nt is head
// slot (8 nt + c) mod 4 NTQ, its hi part (fp16 of the fp32 query) in the first
// half of the columns, its lo part (fp16 of the remainder) in the second;
// slots >= Gv are zero.  q: the sub-group's first query head [Gv][D] fp32,
// in global memory (read through L2: another CTA may have written it in this
// launch) or, with kShared, in this CTA's shared memory.  Items first, first +
// stride, ...
template <int D, int NTQ, bool kShared = false>
__device__ __forceinline__ void build_qfrag(const float* q, int Gv, uint2* qf, int first, int stride) {
  for (int item = first; item < (D / 16) * NTQ * 32; item += stride) {
    const int ln = item & 31, ks = (item >> 5) / NTQ, nt = (item >> 5) - NTQ * ks;
    const int col = 8 * nt + (ln >> 2), part = col / (4 * NTQ), hs = col - part * 4 * NTQ;
    const int k0 = 16 * ks + 2 * (ln & 3);
    uint2 v = make_uint2(0u, 0u);
    if (hs < Gv) {
      const float2* q2 = reinterpret_cast<const float2*>(q + hs * D + k0);
      const float2 f0 = kShared ? q2[0] : __ldcg(q2);
      const float2 f1 = kShared ? q2[4] : __ldcg(q2 + 4);
      uint32_t h0, l0q, h1, l1q;
      split_half2(f0.x, f0.y, h0, l0q);
      split_half2(f1.x, f1.y, h1, l1q);
      v = part ? make_uint2(l0q, l1q) : make_uint2(h0, h1);
    }
    qf[(ks * NTQ + nt) * 32 + ln] = v;
  }
}

// One consumer warp's share of a context: the warp takes the 16-position
// sub-tile `warp` of every 64-position tile and keeps, for this lane's two
// head slots (columns 2t, 2t + 1 of each n-tile; the hi and lo columns of one
// head carry the same slot), the running max m, the normalizer l (a partial
// sum over this lane's positions until finish) and O^T (rows = dims 16 j + g
// (+ 8), columns 2t, 2t + 1).
template <int D, int NTQ>
struct AttnWarp {
  using Lay = AttnLayout<D>;
  float m0, m1, l0, l1;
  float o[D / 16][NTQ][4];

  __device__ __forceinline__ void init() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int j = 0; j < D / 16; ++j)
#pragma unroll
      for (int nt = 0; nt < NTQ; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[j][nt][e] = 0.f;
  }

  // The tile in Ks (key codes, value codes, key scales, value scales; npos of
  // its 64 positions valid).
  __device__ __forceinline__ void tile(const uint8_t* Ks, int npos, const uint2* qf, float qk_scale_log2) {
    const int warp = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const uint8_t* Vs = Ks + Lay::kCodes;
    const __half* ksc = reinterpret_cast<const __half*>(Ks + 2 * Lay::kCodes);
    const __half* vsc = ksc + kTilePos;
    if (16 * warp < npos) {
      // S^T = K q'^T over the D/16 k-steps; even and odd k-steps in two
      // accumulators (shorter MMA chains)
      float sa[NTQ][4], sb[NTQ][4];
#pragma unroll
      for (int nt = 0; nt < NTQ; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
      const uint32_t* kw0 = reinterpret_cast<const uint32_t*>(Ks + (size_t)(2 * warp) * (4 * D) + lane * (D / 8));
      const uint32_t* kw1 = reinterpret_cast<const uint32_t*>(Ks + (size_t)(2 * warp + 1) * (4 * D) + lane * (D / 8));
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        // a code word holds the key's B-operand pairs of k-steps 2j and 2j+1;
        // the two 8-position halves stack into the A operand's 16 rows
        uint32_t c0[4], c1[4];
        nib4_f16x2(kw0[j], c0);
        nib4_f16x2(kw1[j], c1);
        const uint32_t ae[4] = {c0[0], c1[0], c0[1], c1[1]};
        const uint32_t ao[4] = {c0[2], c1[2], c0[3], c1[3]};
#pragma unroll
        for (int nt = 0; nt < NTQ; ++nt) {
          const uint2 qe = qf[((2 * j) * NTQ + nt) * 32 + lane];
          const uint2 qo = qf[((2 * j + 1) * NTQ + nt) * 32 + lane];
          mma_f16_16816(sa[nt], ae, qe.x, qe.y);
          mma_f16_16816(sb[nt], ao, qo.x, qo.y);
        }
      }
      // hi + lo: with one n-tile the lo column of this lane's heads sits in
      // lane t ^ 2; with two, in the second n-tile.  Both lanes of a pair
      // end with the same sums (addition commutes).
      float sv[4];  // [key half][head]: (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (NTQ == 1) {
          const float v = sa[0][e] + sb[0][e];
          sv[e] = v + __shfl_xor_sync(0xffffffffu, v, 2);
        } else {
          sv[e] = (sa[0][e] + sb[0][e]) + (sa[1][e] + sb[1][e]);
        }
      }
      const int pk0 = 16 * warp + g, pk1 = pk0 + 8;
      const bool v0 = pk0 < npos, v1 = pk1 < npos;
      const float ks0 = v0 ? __half2float(ksc[pk0]) * qk_scale_log2 : 0.f;
      const float ks1 = v1 ? __half2float(ksc[pk1]) * qk_scale_log2 : 0.f;
      const float vs0 = v0 ? __half2float(vsc[pk0]) : 0.f;
      const float vs1 = v1 ? __half2float(vsc[pk1]) : 0.f;
      const float sc0 = v0 ? sv[0] * ks0 : -INFINITY, sc1 = v0 ? sv[1] * ks0 : -INFINITY;
      const float sc2 = v1 ? sv[2] * ks1 : -INFINITY, sc3 = v1 ? sv[3] * ks1 : -INFINITY;
      // tile max of each head over the 16 positions (lanes g = 0..7)
      float mx0 = fmaxf(sc0, sc2), mx1 = fmaxf(sc1, sc3);
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float corr0 = mn0 == -INFINITY ? 1.f : ex2_approx(m0 - mn0);
      const float corr1 = mn1 == -INFINITY ? 1.f : ex2_approx(m1 - mn1);
      const float p0 = v0 ? ex2_approx(sc0 - mn0) : 0.f, p1 = v0 ? ex2_approx(sc1 - mn1) : 0.f;
      const float p2 = v1 ? ex2_approx(sc2 - mn0) : 0.f, p3 = v1 ? ex2_approx(sc3 - mn1) : 0.f;
      l0 = l0 * corr0 + (p0 + p2);
      l1 = l1 * corr1 + (p1 + p3);
      m0 = mn0;
      m1 = mn1;
      // rescale O only when some head's running max moved (corr = 1
      // otherwise: the product would leave O unchanged)
      if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {
#pragma unroll
        for (int j = 0; j < D / 16; ++j)
#pragma unroll
          for (int nt = 0; nt < NTQ; ++nt) {
            o[j][nt][0] *= corr0;
            o[j][nt][1] *= corr1;
            o[j][nt][2] *= corr0;
            o[j][nt][3] *= corr1;
          }
      }
      // P^T operand: p * value_scale as an fp16 pair hi + lo (hi = fp16(v),
      // lo = fp16(v - hi)), hi in the first half of the columns; the
      // (position, column) fragment is transposed to (column, position)
      uint32_t ht, lt, hb, lb;
      split_half2(p0 * vs0, p1 * vs0, ht, lt);
      split_half2(p2 * vs1, p3 * vs1, hb, lb);
      uint32_t bt[NTQ], bb[NTQ];
      if (NTQ == 1) {
        bt[0] = movmatrix_trans(t >= 2 ? lt : ht);
        bb[0] = movmatrix_trans(t >= 2 ? lb : hb);
      } else {
        bt[0] = movmatrix_trans(ht);
        bb[0] = movmatrix_trans(hb);
        bt[NTQ - 1] = movmatrix_trans(lt);
        bb[NTQ - 1] = movmatrix_trans(lb);
      }
      const uint32_t* vw = reinterpret_cast<const uint32_t*>(Vs + (size_t)warp * (8 * D) + lane * (D / 4));
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        // a value code word holds the B-operand pairs of dims 16j + g and
        // 16j + 8 + g: as the A operand of V^T they are rows g and g + 8
        uint32_t vv[4];
        nib4_f16x2(vw[j], vv);
        const uint32_t av[4] = {vv[0], vv[2], vv[1], vv[3]};
#pragma unroll
        for (int nt = 0; nt < NTQ; ++nt) mma_f16_16816(o[j][nt], av, bt[nt], bb[nt]);
      }
    }
  }

  // The lane partials summed (l) and the hi + lo columns of O^T added; this
  // warp's (m, l, O) rows to shared memory cm, cl [warps][G], co [warps][G][D]
  // (the lanes with the hi columns write their two heads).
  __device__ __forceinline__ void finish(float* cm, float* cl, float* co, int G, int Gv) {
    const int warp = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
      l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }
    // hi + lo columns of O^T
#pragma unroll
    for (int j = 0; j < D / 16; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (NTQ == 1)
          o[j][0][e] += __shfl_xor_sync(0xffffffffu, o[j][0][e], 2);
        else
          o[j][0][e] += o[j][NTQ - 1][e];
      }

    // this warp's (m, l, O) rows to shared memory: the lanes with the hi
    // columns write their two heads
    const int ha = NTQ == 1 ? 2 * (t & 1) : 2 * t;
    if (NTQ > 1 || t < 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = ha + e;
        if (h < Gv) {
          if (g == 0) {
            cm[warp * G + h] = e ? m1 : m0;
            cl[warp * G + h] = e ? l1 : l0;
          }
#pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            co[(warp * G + h) * D + 16 * j + g] = o[j][0][e];
            co[(warp * G + h) * D + 16 * j + 8 + g] = o[j][0][2 + e];
          }
        }
      }
    }
  }
};

// The consumer warps' (m, l, O) rows merged into (mO [Gv][D], mm, ml [Gv]):
// threads first, first + stride, ... of the caller's group.  The weights of
// each (warp, head), exp2(m_w - M), are computed once per head into
// wbuf [kAttnCW][G] (between two `sync` calls of the whole group), then every
// element adds the warps' rows in warp order.
template <class Sync>
__device__ __forceinline__ void merge_warps(const float* cm, const float* cl, const float* co, float* mO, float* mm,
                                            float* ml, float* wbuf, int G, int Gv, int D, int first, int stride,
                                            Sync&& sync) {
  for (int r = first; r < Gv; r += stride) {
    float M = -INFINITY;
    for (int w = 0; w < kAttnCW; ++w) M = fmaxf(M, cm[w * G + r]);
    float Lr = 0.f;
    for (int w = 0; w < kAttnCW; ++w) {
      const float mw = cm[w * G + r];
      const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
      wbuf[w * G + r] = wt;
      Lr += cl[w * G + r] * wt;
    }
    mm[r] = M;
    ml[r] = Lr;
  }
  sync();
  for (int e = first; e < Gv * D; e += stride) {
    const int r = e / D, i = e % D;
    float Or = 0.f;
    for (int w = 0; w < kAttnCW; ++w) Or += co[(w * G + r) * D + i] * wbuf[w * G + r];
    mO[e] = Or;
  }
}

}  // namespace
}  // namespace futr
