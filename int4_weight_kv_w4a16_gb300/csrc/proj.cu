// W4A16 decode projection: y = W' x with INT4 weights and bf16 activations.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract and explainer section "INT4 Decode: letting
// dequantization feed directly into MMA operands": the packed nibbles are
// converted in registers straight into mma.m16n8k16 A fragments (weights are
// the M side, the batch of 1..32 tokens the N side), without a dequantized
// tile in memory.  The codes enter the MMA exactly; each 128-input group's
// fp32 partial sum is multiplied by its fp16 scale afterwards.
//
// Structure of one CTA (row block of 128 outputs x a K-range of groups):
//   warp 8 (producer): 1-D bulk copies of 8448-byte units (codes + scales)
//     into a ring of shared-memory stages, completion tracked by mbarriers;
//     the first stages are issued before griddepcontrol.wait so that weight
//     streaming overlaps the previous kernel.  After the wait it also copies
//     the CTA's activation slice [batch][K-range].
//   warps 0..7 (consumers): warp w owns rows 16w..16w+15; per group it reads
//     its 32 bytes of nibbles and two scales, releases the stage, builds the
//     B fragments with ldmatrix from the activation slice and issues 8*NT mma.
//   split-K: each CTA writes a partial [batch][128] (+ sum of squares of its
//     activation slice, for RMSNorm); the last CTA of a row block (arrival
//     counter, no spinning) adds the partials in fixed order and runs the
//     epilogue:
//     RESID : out = bf16(resid + acc)                      (O, down)
//     SWIGLU: a = bf16(silu(r g) * (r u)), r = rms factor  (gate/up rows
//             interleaved 64/64 per row block)
//     QKV   : r * acc, RoPE(q, k) at pos, fp32 Hadamard rotation; q -> fp32
//             rotated query; k, v -> INT4 + fp16 scale into cache slot pos
//             (direct KV-cache placement, abstract).
#include "futr_internal.cuh"
#include "proj.cuh"

namespace futr {

namespace {

constexpr int kCW = 8;                    // consumer warps
constexpr int kThreads = (kCW + 1) * 32;  // + producer warp

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
}

template <int J>
__device__ void qkv_head_epilogue(const ProjArgs& a, const float* red, int n, int hl, int hg, float r) {
  constexpr int d = 32 * J;
  const int lane = threadIdx.x & 31;
  float v[J];
#pragma unroll
  for (int j = 0; j < J; ++j) v[j] = red[n * kRedLd + hl * d + lane + 32 * j] * r;
  const int p = a.pos[n];
  const bool is_q = hg < a.Hq, is_k = !is_q && hg < a.Hq + a.Hkv;
  const bool p_ok = p >= 0 && p < a.kv.cap;
  if (is_q || is_k) {
    // rotate-half RoPE: dims i and i + d/2 (lane-local: element j pairs j + J/2)
    const int pp = p_ok ? p : 0;
#pragma unroll
    for (int j = 0; j < J / 2; ++j) {
      const float2 cs = a.rope[(size_t)pp * (d / 2) + lane + 32 * j];
      const float x1 = v[j], x2 = v[j + J / 2];
      v[j] = x1 * cs.x - x2 * cs.y;
      v[j + J / 2] = x2 * cs.x + x1 * cs.y;
    }
  }
  warp_fwht<J>(v, a.nh, a.had_c);
  if (is_q) {
    float* q = a.qrot + ((size_t)n * a.Hq + hg) * d;
#pragma unroll
    for (int j = 0; j < J; ++j) q[lane + 32 * j] = v[j];
    return;
  }
  int code[J];
  const __half s = warp_quant<J>(v, code);
  if (!p_ok) {
    if (lane == 0) set_err(a.err, FUTR_ERR_OUT_OF_RANGE);
    return;
  }
  __shared__ int8_t scratch[kCW][d];
  const int warp = threadIdx.x >> 5;
  if (is_k)
    store_k_token<J>(a.kv.stream(n, hg - a.Hq), a.kv.cap, p, code, s, scratch[warp]);
  else
    store_v_token<J>(a.kv.stream(n, hg - a.Hq - a.Hkv), a.kv.cap, p, code, s, scratch[warp]);
}

template <int NT, int EPI>
__global__ void __launch_bounds__(kThreads) proj_kernel(const ProjArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.x / a.S, sk = blockIdx.x - rb * a.S;
  const int g0 = (int)(((long long)sk * a.n_groups) / a.S);
  const int g1 = (int)(((long long)(sk + 1) * a.n_groups) / a.S);
  const int ng = g1 - g0, krange = ng * kGroup, xstride = krange + 8;

  uint8_t* stages = smem;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem + a.off_xs);
  float* ss = reinterpret_cast<float*>(smem + a.off_misc);  // [32] sum of squares per batch row
  float* wsum = ss + 32;                                      // [kCW][32]
  int* flag = reinterpret_cast<int*>(wsum + kCW * 32);        // [4]
  uint64_t* full = reinterpret_cast<uint64_t*>(flag + 4);
  uint64_t* empty = full + kStages;
  uint64_t* xbar = empty + kStages;
  float* red = reinterpret_cast<float*>(smem);  // epilogue [NT*8][kRedLd], aliases the stages

  if (tid == 0) {
    flag[0] = 0;
    flag[1] = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    mbar_init(xbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();

  const uint8_t* unit0 = a.w + ((size_t)rb * a.n_groups + g0) * kUnitBytes;
  if (warp == kCW) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const int pre = ng < kStages ? ng : kStages;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], kUnitBytes);
        bulk_g2s(stages + i * kUnitBytes, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[i]);
      }
      pdl_wait();
      const unsigned long long deadline = global_ns() + kWaitNs;
      mbar_arrive_expect_tx(xbar, (uint32_t)(a.batch * krange * 2));
      for (int n = 0; n < a.batch; ++n)
        bulk_g2s(xs + n * xstride, a.xin + (size_t)n * a.K + (size_t)g0 * kGroup, krange * 2, xbar);
      for (int i = kStages; i < ng; ++i) {
        const int slot = i % kStages;
        if (!mbar_wait_until(&empty[slot], ((i / kStages) - 1) & 1, deadline)) {
          set_err(a.err, FUTR_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[slot], kUnitBytes);
        bulk_g2s(stages + slot * kUnitBytes, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[slot]);
      }
    } else {
      pdl_wait();
    }
    return;
  }

  // ----------------------------------------------------------- consumers --
  pdl_wait();
  const unsigned long long deadline = global_ns() + kWaitNs;
  bool ok = mbar_wait_until(xbar, 0, deadline);

  if (EPI != kEpiResid) {
    // sum of squares of this CTA's activation slice, fixed reduction order
    for (int n = 0; n < a.batch; ++n) {
      float acc = 0.f;
      for (int c = tid; c < krange; c += kCW * 32) {
        const float x = __bfloat162float(xs[n * xstride + c]);
        acc = fmaf(x, x, acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) wsum[warp * 32 + n] = acc;
    }
  }
  consumer_sync();
  if (EPI != kEpiResid && tid < a.batch) {
    float acc = 0.f;
    for (int w = 0; w < kCW; ++w) acc += wsum[w * 32 + tid];
    ss[tid] = acc;
  }

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

  const int rt = warp, gr = lane >> 2;
  // ldmatrix row addresses of this lane: batch row 8nt + (lane & 7), column
  // block (lane >> 3).  Rows past the batch read row 0 instead: they only feed
  // MMA columns that are never stored.
  const __nv_bfloat16* xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = 8 * nt + (lane & 7);
    xrow[nt] = xs + (n < a.batch ? n : 0) * xstride + 8 * (lane >> 3);
  }
  for (int i = 0; i < ng; ++i) {
    const int slot = i % kStages;
    if (!mbar_wait_until(&full[slot], (i / kStages) & 1, deadline)) {
      ok = false;
      break;
    }
    const uint8_t* st = stages + slot * kUnitBytes;
    const uint4* wt = reinterpret_cast<const uint4*>(st + rt * 1024);
    const uint4 w0 = wt[lane], w1 = wt[32 + lane];
    const __half* sc = reinterpret_cast<const __half*>(st + kUnitCodeBytes);
    const float s_lo = __half2float(sc[rt * 16 + gr]), s_hi = __half2float(sc[rt * 16 + gr + 8]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);

    float dpart[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) dpart[nt][e] = 0.f;
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      uint32_t bfr[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) ldmatrix_x4(bfr[nt], xrow[nt] + i * kGroup + 32 * kp);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w = words[2 * kp + h];
        const uint32_t af[4] = {nib_bf16x2(w, 0), nib_bf16x2(w, 1), nib_bf16x2(w, 2), nib_bf16x2(w, 3)};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(dpart[nt], af, bfr[nt][2 * h], bfr[nt][2 * h + 1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[nt][0] = fmaf(s_lo, dpart[nt][0], acc[nt][0]);
      acc[nt][1] = fmaf(s_lo, dpart[nt][1], acc[nt][1]);
      acc[nt][2] = fmaf(s_hi, dpart[nt][2], acc[nt][2]);
      acc[nt][3] = fmaf(s_hi, dpart[nt][3], acc[nt][3]);
    }
  }
  if (!ok) {
    set_err(a.err, FUTR_ERR_TIMEOUT);
    flag[1] = 1;
  }

  // ------------------------------------------------------------ epilogue --
  consumer_sync();  // every warp is done with the stage ring: reuse it as `red`
  if (flag[1]) return;  // a wait ran out: the ring may still be in use, write nothing
  {
    const int t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n0 = 8 * nt + 2 * t;
      red[n0 * kRedLd + 16 * rt + gr] = acc[nt][0];
      red[(n0 + 1) * kRedLd + 16 * rt + gr] = acc[nt][1];
      red[n0 * kRedLd + 16 * rt + gr + 8] = acc[nt][2];
      red[(n0 + 1) * kRedLd + 16 * rt + gr + 8] = acc[nt][3];
    }
  }
  consumer_sync();

  if (a.S > 1) {
    // publish this split's partial, then count arrivals; the last CTA reduces
    float* rec = a.part + ((size_t)rb * a.S + sk) * a.rec_floats;
    for (int e = tid; e < a.batch * 32; e += kCW * 32) {
      const int n = e >> 5, c4 = e & 31;
      reinterpret_cast<float4*>(rec + n * kRowsPerBlock)[c4] = reinterpret_cast<const float4*>(red + n * kRedLd)[c4];
    }
    if (tid < a.batch) rec[a.batch * kRowsPerBlock + tid] = ss[tid];
    __threadfence();
    consumer_sync();
    if (tid == 0) {
      const unsigned prev = atomicAdd(&a.cnt[rb], 1u);
      flag[0] = (prev == (unsigned)(a.S - 1)) ? 1 : 0;
    }
    consumer_sync();
    if (!flag[0]) return;
    __threadfence();
    // add the S partials in split order, 8 independent loads in flight
    const float* part_rb = a.part + (size_t)rb * a.S * a.rec_floats;
    for (int e = tid; e < a.batch * 32; e += kCW * 32) {
      const int n = e >> 5, c4 = e & 31;
      float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < a.S; s0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < a.S)
            v[j] = __ldcg(reinterpret_cast<const float4*>(part_rb + (size_t)(s0 + j) * a.rec_floats +
                                                          n * kRowsPerBlock) + c4);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < a.S) {
            s4.x += v[j].x; s4.y += v[j].y; s4.z += v[j].z; s4.w += v[j].w;
          }
      }
      reinterpret_cast<float4*>(red + n * kRedLd)[c4] = s4;
    }
    if (tid < a.batch) {
      float s2 = 0.f;
      for (int s0 = 0; s0 < a.S; s0 += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[j] = s0 + j < a.S ? __ldcg(part_rb + (size_t)(s0 + j) * a.rec_floats + a.batch * kRowsPerBlock + tid) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < a.S) s2 += v[j];
      }
      ss[tid] = s2;
    }
    if (tid == 0) a.cnt[rb] = 0u;  // self-reset for the next launch
    consumer_sync();
  }

  if (EPI == kEpiResid) {
    for (int e = tid; e < a.batch * kRowsPerBlock; e += kCW * 32) {
      const int n = e >> 7, r = e & 127;
      const size_t o = (size_t)n * a.out_ld + (size_t)rb * kRowsPerBlock + r;
      a.out[o] = __float2bfloat16_rn(__bfloat162float(a.resid[o]) + red[n * kRedLd + r]);
    }
  } else if (EPI == kEpiSwiglu) {
    for (int e = tid; e < a.batch * 64; e += kCW * 32) {
      const int n = e >> 6, r = e & 63;
      const float rn = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(ss[n], (float)a.K) + a.eps));
      const float g = rn * red[n * kRedLd + r];
      const float u = rn * red[n * kRedLd + 64 + r];
      const float sg = __fdiv_rn(g, 1.0f + expf(-g));
      a.out[(size_t)n * a.out_ld + (size_t)rb * 64 + r] = __float2bfloat16_rn(sg * u);
    }
  } else {
    if (rb == 0 && tid == 0 && a.blob_magic && *a.blob_magic != kBlobMagic)
      set_err(a.err, FUTR_ERR_BAD_BLOB);
    const int hpr = kRowsPerBlock / a.d;
    for (int task = warp; task < a.batch * hpr; task += kCW) {
      const int n = task / hpr, hl = task % hpr;
      const int hg = rb * hpr + hl;
      const float rn = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(ss[n], (float)a.K) + a.eps));
      if (a.d == 128)
        qkv_head_epilogue<4>(a, red, n, hl, hg, rn);
      else
        qkv_head_epilogue<2>(a, red, n, hl, hg, rn);
    }
  }
}

template <int NT, int EPI>
cudaError_t launch_one(const ProjArgs& a, int grid, size_t smem, cudaStream_t st, bool pdl) {
  static unsigned long long configured = 0;  // one bit per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(proj_kernel<NT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kProjMaxSmem);
    if (e != cudaSuccess) return e;
    // every kernel of the step asks for the maximum shared-memory carveout, so
    // CTAs of consecutive kernels can share an SM (programmatic overlap)
    e = cudaFuncSetAttribute(proj_kernel<NT, EPI>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured |= 1ull << (dev & 63);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, proj_kernel<NT, EPI>, a);
}

template <int EPI>
cudaError_t launch_nt(int nt, const ProjArgs& a, int grid, size_t smem, cudaStream_t st, bool pdl) {
  switch (nt) {
    case 1: return launch_one<1, EPI>(a, grid, smem, st, pdl);
    case 2: return launch_one<2, EPI>(a, grid, smem, st, pdl);
    case 3: return launch_one<3, EPI>(a, grid, smem, st, pdl);
    default: return launch_one<4, EPI>(a, grid, smem, st, pdl);
  }
}

}  // namespace

ProjPlan plan_projection(int rows, int cols, int batch, int n_sm, int force_split) {
  ProjPlan p;
  p.n_rb = rows / kRowsPerBlock;
  p.n_groups = cols / kGroup;
  p.nt = (batch + 7) / 8;
  // activation slice limit: NT*8 rows of (groups*128 + 8) bf16 within kXsMax bytes
  const int max_groups = ((kXsMax / (batch * 2)) - 8) / kGroup;
  const int s_min = (p.n_groups + max_groups - 1) / max_groups;
  int s = (2 * n_sm + p.n_rb - 1) / p.n_rb;
  if (force_split > 0) s = force_split;
  if (s < s_min) s = s_min;
  if (s > p.n_groups) s = p.n_groups;
  if (s < 1) s = 1;
  p.S = s;
  const int gmax = (p.n_groups + s - 1) / s;
  p.off_xs = kStages * kUnitBytes;
  int xs_bytes = ((batch * (gmax * kGroup + 8) * 2) + 127) & ~127;
  const int red_bytes = p.nt * 8 * kRedLd * 4;  // the epilogue tile aliases stages + slice
  if (kStages * kUnitBytes + xs_bytes < red_bytes) xs_bytes = red_bytes - kStages * kUnitBytes;
  p.off_misc = p.off_xs + xs_bytes;
  p.smem = p.off_misc + (32 + kCW * 32) * 4 + 16 + (2 * kStages + 1) * 8;
  p.rec_floats = ((batch * (kRowsPerBlock + 1)) + 3) & ~3;
  p.part_floats = (size_t)p.n_rb * p.S * p.rec_floats;
  return p;
}

cudaError_t launch_projection(int epi, const ProjPlan& p, ProjArgs a, cudaStream_t st, bool pdl) {
  a.S = p.S;
  a.n_groups = p.n_groups;
  a.off_xs = p.off_xs;
  a.off_misc = p.off_misc;
  a.rec_floats = p.rec_floats;
  const int grid = p.n_rb * p.S;
  if (epi == kEpiResid) return launch_nt<kEpiResid>(p.nt, a, grid, p.smem, st, pdl);
  if (epi == kEpiSwiglu) return launch_nt<kEpiSwiglu>(p.nt, a, grid, p.smem, st, pdl);
  return launch_nt<kEpiQkv>(p.nt, a, grid, p.smem, st, pdl);
}

}  // namespace futr
