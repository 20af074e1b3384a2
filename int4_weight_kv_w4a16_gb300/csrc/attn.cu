// Single-query GQA decode attention over the INT4 rotated KV cache.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract: decode reads an INT4 KV-cache copy whose keys follow the
// Tensor Core fragment layout; a block-diagonal Hadamard transform is applied
// to the cache, and (explainer, Hadamard paragraph) correspondingly before and
// after: the query is rotated the same way (in the QKV epilogue) and the
// attention output is rotated back here.
//
// One CTA = (sequence b, kv-head, chunk of CH positions); 4 warps take the
// chunk's 16-position tiles in turn.  Per tile a warp runs
//   S = q' K^T: mma.m16n8k16 f16, A = the G query heads of this kv-head
//     (rows >= G are zero) as an fp16 pair hi + lo of the fp32 query (two
//     MMAs), B = key codes converted in registers (exact);
//     score = S * key_scale * log2(e)/sqrt(d);
//   online softmax in fp32 (running max m, normalizer l, output rescale);
//   O += P V: A = fp16(p * value_scale) straight from the score registers,
//     B = value codes converted in registers.
// The 4 warps merge in shared memory; with several chunks, each writes
// (m, l, O) and the last CTA of (b, kv-head) merges them in chunk order, then
// divides by l, undoes the rotation (fp32 Hadamard) and stores bf16.
#include "futr_internal.cuh"
#include "proj.cuh"

namespace futr {

namespace {

constexpr int kAttnWarps = 4;

template <int D>
__global__ void __launch_bounds__(kAttnWarps * 32) attn_kernel(const AttnArgs a) {
  constexpr int J = D / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bar;
  __shared__ int flag;
  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int G = a.G, CH = a.CH, cap = a.kv.cap;

  pdl_trigger();
  pdl_wait();  // q' and the new token's cache entries come from the previous kernel
  const int p = a.pos[b];
  if (p < 0 || p >= cap) {
    if (chunk == 0) {
      for (int e = tid; e < G * D; e += kAttnWarps * 32)
        a.out[((size_t)b * a.Hq + kvh * G) * D + e] = __float2bfloat16_rn(0.f);
      if (kvh == 0 && tid == 0) set_err(a.err, FUTR_ERR_OUT_OF_RANGE);
    }
    return;
  }
  const int L = p + 1, n_chunks = (L + CH - 1) / CH;
  if (chunk >= n_chunks) return;
  const int c0 = chunk * CH, npos = min(CH, L - c0), ntile = (npos + 15) / 16;

  uint8_t* Ks = smem;
  uint8_t* Vs = Ks + (size_t)CH * (D / 2);
  __half* ksc = reinterpret_cast<__half*>(Vs + (size_t)CH * (D / 2));
  __half* vsc = ksc + CH;
  float* cm = reinterpret_cast<float*>(vsc + CH);  // [warps][G]
  float* cl = cm + kAttnWarps * G;                  // [warps][G]
  float* co = cl + kAttnWarps * G;                  // [warps][G][D]
  float* mo = co + kAttnWarps * G * D;              // merged [G][D] O, [G] m, [G] l (16-B aligned)

  const uint8_t* strm = a.kv.stream(b, kvh);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    flag = 0;
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t cb = (uint32_t)ntile * 16 * (D / 2), sb = (uint32_t)ntile * 32;
    mbar_arrive_expect_tx(&bar, 2 * cb + 2 * sb);
    bulk_g2s(Ks, strm + (size_t)c0 * (D / 2), cb, &bar);
    bulk_g2s(Vs, strm + (size_t)cap * (D / 2) + (size_t)c0 * (D / 2), cb, &bar);
    bulk_g2s(ksc, strm + (size_t)cap * D + 2 * (size_t)c0, sb, &bar);
    bulk_g2s(vsc, strm + (size_t)cap * D + 2 * (size_t)cap + 2 * (size_t)c0, sb, &bar);
  }

  // query fragments (A operand of q.k): rows = heads of this group, padded to
  // 16; each fp32 pair becomes fp16 hi + lo registers
  uint32_t qa[D / 16][4], ql[D / 16][4];
  {
    const float* q = a.qrot + ((size_t)b * a.Hq + (size_t)kvh * G) * D;
    const float2 zero = make_float2(0.f, 0.f);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c = 16 * ks + 2 * t;
      const float2 f0 = g < G ? *reinterpret_cast<const float2*>(q + g * D + c) : zero;
      const float2 f1 = g + 8 < G ? *reinterpret_cast<const float2*>(q + (g + 8) * D + c) : zero;
      const float2 f2 = g < G ? *reinterpret_cast<const float2*>(q + g * D + c + 8) : zero;
      const float2 f3 = g + 8 < G ? *reinterpret_cast<const float2*>(q + (g + 8) * D + c + 8) : zero;
      split_half2(f0.x, f0.y, qa[ks][0], ql[ks][0]);
      split_half2(f1.x, f1.y, qa[ks][1], ql[ks][1]);
      split_half2(f2.x, f2.y, qa[ks][2], ql[ks][2]);
      split_half2(f3.x, f3.y, qa[ks][3], ql[ks][3]);
    }
  }
  const bool ok = mbar_wait_until(&bar, 0, global_ns() + kWaitNs);
  if (__syncthreads_or(!ok)) {  // CTA-uniform decision
    if (tid == 0) set_err(a.err, FUTR_ERR_TIMEOUT);
    return;
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nd][e] = 0.f;

  for (int tt = warp; tt < ntile; tt += kAttnWarps) {
    float s[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[h][e] = 0.f;
      const uint32_t* kw = reinterpret_cast<const uint32_t*>(Ks + (size_t)(2 * tt + h) * (4 * D) + lane * (D / 8));
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        const uint32_t w = kw[j];
        const uint32_t k0 = nib_f16x2(w, 0), k1 = nib_f16x2(w, 1), k2 = nib_f16x2(w, 2), k3 = nib_f16x2(w, 3);
        mma_f16_16816(s[h], qa[2 * j], k0, k1);
        mma_f16_16816(s[h], qa[2 * j + 1], k2, k3);
        mma_f16_16816(s[h], ql[2 * j], k0, k1);
        mma_f16_16816(s[h], ql[2 * j + 1], k2, k3);
      }
    }
    float sc[2][4], vsv[2][2];
    bool valid[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int pl = 16 * tt + 8 * h + 2 * t + e;
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
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o[nd][0] *= corr0;
      o[nd][1] *= corr0;
      o[nd][2] *= corr1;
      o[nd][3] *= corr1;
    }
    // P operand = p * value_scale as an fp16 pair hi + lo (hi = fp16(v),
    // lo = fp16(v - hi)): two MMAs keep ~22 bits of each weight.
    uint32_t pa[4], pl[4];
    split_half2(pr[0][0] * vsv[0][0], pr[0][1] * vsv[0][1], pa[0], pl[0]);
    split_half2(pr[0][2] * vsv[0][0], pr[0][3] * vsv[0][1], pa[1], pl[1]);
    split_half2(pr[1][0] * vsv[1][0], pr[1][1] * vsv[1][1], pa[2], pl[2]);
    split_half2(pr[1][2] * vsv[1][0], pr[1][3] * vsv[1][1], pa[3], pl[3]);
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(Vs + (size_t)tt * (8 * D) + lane * (D / 4));
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const uint32_t w = vw[j];
      const uint32_t v0 = nib_f16x2(w, 0), v1 = nib_f16x2(w, 1), v2 = nib_f16x2(w, 2), v3 = nib_f16x2(w, 3);
      mma_f16_16816(o[2 * j], pa, v0, v1);
      mma_f16_16816(o[2 * j + 1], pa, v2, v3);
      mma_f16_16816(o[2 * j], pl, v0, v1);
      mma_f16_16816(o[2 * j + 1], pl, v2, v3);
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- merge the 4 warps
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
  __syncthreads();
  float* mO = mo;
  float* mm = mo + G * D;
  float* ml = mm + G;
  for (int e = tid; e < G * D; e += kAttnWarps * 32) {
    const int r = e / D, i = e % D;
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, cm[w * G + r]);
    float Lr = 0.f, Or = 0.f;
    for (int w = 0; w < kAttnWarps; ++w) {
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

  if (n_chunks > 1) {
    const size_t rec_base = (((size_t)b * a.Hkv + kvh) * a.max_chunks) * a.rec_floats;
    float* rec = a.apart + rec_base + (size_t)chunk * a.rec_floats;
    for (int e = tid; e < G * (D + 2); e += kAttnWarps * 32) rec[e] = mo[e];
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned prev = atomicAdd(&a.cnt[b * a.Hkv + kvh], 1u);
      flag = prev == (unsigned)(n_chunks - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!flag) return;
    __threadfence();
    // merge the chunks in chunk order: (m, l) of every chunk to shared memory,
    // per-chunk weights exp2(m_c - M), then O with independent loads in flight
    float* wm = co;                   // [n_chunks][G] m, then weights
    float* wl = co + n_chunks * G;    // [n_chunks][G] l
    for (int i = tid; i < n_chunks * G; i += kAttnWarps * 32) {
      const float* rc = a.apart + rec_base + (size_t)(i / G) * a.rec_floats;
      wm[i] = __ldcg(rc + G * D + i % G);
      wl[i] = __ldcg(rc + G * D + G + i % G);
    }
    __syncthreads();
    if (tid < G) {
      float M = -INFINITY;
      for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, wm[c * G + tid]);
      float Lr = 0.f;
      for (int c = 0; c < n_chunks; ++c) {
        const float wt = exp2f(wm[c * G + tid] - M);
        wm[c * G + tid] = wt;
        Lr += wl[c * G + tid] * wt;
      }
      ml[tid] = Lr;
    }
    __syncthreads();
    // four consecutive elements per thread (float4); 8 chunk loads in flight
    for (int e4 = tid; e4 < G * D / 4; e4 += kAttnWarps * 32) {
      const int r = (4 * e4) / D;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      const float* src = a.apart + rec_base + 4 * e4;
      for (int c0 = 0; c0 < n_chunks; c0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[j] = c0 + j < n_chunks ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)(c0 + j) * a.rec_floats))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float wt = c0 + j < n_chunks ? wm[(c0 + j) * G + r] : 0.f;
          acc.x += v[j].x * wt; acc.y += v[j].y * wt; acc.z += v[j].z * wt; acc.w += v[j].w * wt;
        }
      }
      reinterpret_cast<float4*>(mO)[e4] = acc;
    }
    if (tid == 0) a.cnt[b * a.Hkv + kvh] = 0u;
    __syncthreads();
  }

  // ---- normalize, rotate back, store bf16
  for (int r = warp; r < G; r += kAttnWarps) {
    const float inv = __fdiv_rn(1.0f, ml[r]);
    float v[J];
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] = mO[r * D + lane + 32 * j] * inv;
    warp_fwht<J>(v, a.nh, a.had_c);
    __nv_bfloat16* out = a.out + ((size_t)b * a.Hq + (size_t)kvh * G + r) * D;
#pragma unroll
    for (int j = 0; j < J; ++j) out[lane + 32 * j] = __float2bfloat16_rn(v[j]);
  }
}

template <int D>
cudaError_t launch_d(const AttnPlan& p, const AttnArgs& a, cudaStream_t st, bool pdl) {
  static unsigned long long configured = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured |= 1ull << (dev & 63);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.max_chunks, (unsigned)a.Hkv, (unsigned)a.batch);
  cfg.blockDim = dim3(kAttnWarps * 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_kernel<D>, a);
}

}  // namespace

AttnPlan plan_attention(const futr_shape& s, int batch, int cap, int n_sm, int force_chunk) {
  AttnPlan p;
  const int G = s.n_q_heads / s.n_kv_heads, D = s.head_dim;
  int ch = 64;
  while (ch < 512 && (long long)batch * s.n_kv_heads * ((cap + ch - 1) / ch) > 8LL * n_sm) ch *= 2;
  if (force_chunk > 0) ch = force_chunk;
  // the last CTA keeps (m, l) of every chunk in 4*G*D floats of shared memory
  while ((cap + ch - 1) / ch > 2 * D) ch *= 2;
  p.CH = ch;
  p.max_chunks = (cap + ch - 1) / ch;
  p.rec_floats = (G * (D + 2) + 3) & ~3;
  p.part_floats = (size_t)batch * s.n_kv_heads * p.max_chunks * p.rec_floats;
  p.smem = (size_t)ch * D + 4 * (size_t)ch + (size_t)(2 * kAttnWarps * G + kAttnWarps * G * D) * 4 +
           (size_t)(2 * G + G * D) * 4;
  return p;
}

cudaError_t launch_attention(const AttnPlan& p, AttnArgs a, int d, cudaStream_t st, bool pdl) {
  a.CH = p.CH;
  a.max_chunks = p.max_chunks;
  a.rec_floats = p.rec_floats;
  return d == 128 ? launch_d<128>(p, a, st, pdl) : launch_d<64>(p, a, st, pdl);
}

}  // namespace futr
