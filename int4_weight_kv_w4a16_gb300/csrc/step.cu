// The rest of a full decode step around the blocks: embedding gather, final
// RMSNorm and the bf16 LM head.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract: the complete Llama-3.1-8B decode step (all blocks plus
// the embedding, the final norm and the LM head).  No INT4 projection follows
// the final norm, so its gain cannot be folded into INT4 codes: the LM head
// stays bf16 and the gain multiplies the last block's output,
//   logits[b, v] = r_b * sum_k W[v, k] * bf16(g_k * y_bk),
//   r_b = 1 / sqrt(mean_k y_bk^2 + eps)   (applied to the fp32 logits).
//
// LM head: CTA = 64 vocabulary rows (4 consumer warps x 16) x all inputs.  A
// producer warp streams 64-row x 64-input boxes of the head (8 KB) and the
// matching 64-input box of the activation (8 rows per batch tile, rows past
// the batch zero-filled by the copy) with 2-D tensor copies (128-byte
// swizzle) into a ring of shared-memory stages; consumers read A and B
// fragments with ldmatrix and accumulate bf16 mma.sync in fp32.
#include <cuda.h>

#include "futr_internal.cuh"

namespace futr {

namespace {

constexpr int kLmRows = 64;                  // vocabulary rows per CTA
constexpr int kLmK = 64;                     // inputs per stage: one 128-byte line per row
constexpr int kLmRing = 6;
constexpr int kLmCW = 4;                     // consumer warps
constexpr int kLmThreads = (kLmCW + 1) * 32;
constexpr int kLmWBytes = kLmRows * kLmK * 2;  // 8192

struct LmArgs {
  const float* r;     // [batch] RMSNorm factors
  float* logits;      // [batch][vocab]
  int vocab, H, batch;
  int* err;
};

__global__ void __launch_bounds__(256) embed_kernel(const int* tokens, const __nv_bfloat16* table, int vocab,
                                                    int H, __nv_bfloat16* x, int* err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int t = tokens[b];
  const bool ok = t >= 0 && t < vocab;
  if (!ok && threadIdx.x == 0) set_err(err, FUTR_ERR_OUT_OF_RANGE);
  const uint4* src = reinterpret_cast<const uint4*>(table + (size_t)(ok ? t : 0) * H);
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)b * H);
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0u, 0u, 0u, 0u);
}

// xg = bf16(fp32(g * y)), r = 1/sqrt(mean(y^2) + eps); one CTA per sequence,
// the sum of squares in a fixed order (deterministic).
__global__ void __launch_bounds__(256) final_norm_kernel(const __nv_bfloat16* y, const float* g, int H, float eps,
                                                         __nv_bfloat16* xg, float* r) {
  __shared__ float part[8];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  float s = 0.f;
  for (int i = tid; i < H; i += 256) {
    const float v = __bfloat162float(y[(size_t)b * H + i]);
    s = fmaf(v, v, s);
    xg[(size_t)b * H + i] = __float2bfloat16_rn(v * g[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((tid & 31) == 0) part[tid >> 5] = s;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += part[w];
    r[b] = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(t, (float)H) + eps));
  }
}

// Shared address of 16-byte chunk c of row r in a box of 128-byte rows
// written with the 128-byte swizzle (chunk index XOR row mod 8; the box
// starts on a 1024-byte boundary).
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <int NT>
__global__ void __launch_bounds__(kLmThreads) lm_head_kernel(const __grid_constant__ CUtensorMap tw,
                                                             const __grid_constant__ CUtensorMap tx, const LmArgs a) {
  constexpr int kXBytes = 8 * NT * kLmK * 2;  // 1024 per batch tile
  constexpr int kStage = kLmWBytes + kXBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kLmRing * kStage);
  uint64_t* empty = full + kLmRing;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = blockIdx.x * kLmRows, n_st = a.H / kLmK;

  // the producer's issued-stage count and stop flag, for the drain after a time-out
  __shared__ int s_issued, s_stopped;
  if (tid == 0) {
    for (int i = 0; i < kLmRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kLmCW);
    }
    fence_mbar_init();
    s_issued = 0;
    s_stopped = 0;
  }
  __syncthreads();
  pdl_trigger();

  if (warp == kLmCW) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const int pre = n_st < kLmRing ? n_st : kLmRing;
      for (int i = 0; i < pre; ++i) {  // head boxes do not depend on the previous kernel
        mbar_arrive_expect_tx(&full[i], kStage);
        tma_2d(smem_u32(smem + i * kStage), &tw, i * kLmK, row0, &full[i]);
      }
      pdl_wait();  // the activation comes from the previous kernel
      const unsigned long long deadline = global_ns() + kWaitNs;
      for (int i = 0; i < pre; ++i) tma_2d(smem_u32(smem + i * kStage + kLmWBytes), &tx, i * kLmK, 0, &full[i]);
      int slot = 0, issued = pre;
      uint32_t phase = 0;
      for (int i = kLmRing; i < n_st; ++i) {
        if (!mbar_wait_until(&empty[slot], phase, deadline, a.err)) {
          record_timeout(a.err);
          break;
        }
        uint8_t* st = smem + slot * kStage;
        mbar_arrive_expect_tx(&full[slot], kStage);
        tma_2d(smem_u32(st), &tw, i * kLmK, row0, &full[slot]);
        tma_2d(smem_u32(st + kLmWBytes), &tx, i * kLmK, 0, &full[slot]);
        issued = i + 1;
        if (++slot == kLmRing) {
          slot = 0;
          phase ^= 1u;
        }
      }
      *reinterpret_cast<volatile int*>(&s_issued) = issued;
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&s_stopped) = 1;
    } else {
      pdl_wait();
    }
    return;
  }

  // ----------------------------------------------------------- consumers --
  pdl_wait();
  const unsigned long long deadline = global_ns() + kWaitNs;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  // A (head rows): ldmatrix matrix m = lane >> 3 is rows (m & 1) * 8 .. +7 of
  // this warp's 16, chunk (m >> 1) of the k-step; B (activation): rows of
  // batch tile nt, chunk m of a 32-input span.
  const int ar = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1), ac = lane >> 4;
  const int xr = lane & 7, xc = lane >> 3;
  int slot = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int i = 0; i < n_st; ++i) {
    if (!mbar_wait_until(&full[slot], phase, deadline, a.err)) {
      ok = false;
      break;
    }
    const uint32_t sw = smem_u32(smem + slot * kStage), sx = sw + kLmWBytes;
#pragma unroll
    for (int kp = 0; kp < 2; ++kp) {
      uint32_t bfr[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) ldsm_x4(bfr[nt], swz(sx, 8 * nt + xr, 4 * kp + xc));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t af[4];
        ldsm_x4(af, swz(sw, ar, 2 * (2 * kp + h) + ac));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt], af, bfr[nt][2 * h], bfr[nt][2 * h + 1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (++slot == kLmRing) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (!ok) {
    // let the producer stop and the copies it issued land before leaving
    record_timeout(a.err);
    if (lane == 0) {
      const unsigned long long dl = global_ns() + kWaitNs;
      while (*reinterpret_cast<volatile int*>(&s_stopped) == 0 && global_ns() < dl) {
      }
      __threadfence_block();
      drain_ring(full, kLmRing, *reinterpret_cast<volatile int*>(&s_issued));
    }
    __syncwarp();
    return;
  }
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = 8 * nt + 2 * t + (e & 1);
      const int row = row0 + 16 * warp + g + 8 * (e >> 1);
      if (n < a.batch) a.logits[(size_t)n * a.vocab + row] = a.r[n] * acc[nt][e];
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 row-major [outer][inner] tensor, boxes of box_outer x 64 elements
// (128-byte rows, 128-byte swizzle); out-of-range rows read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kLmK, box_outer};
  const cuuint32_t elem[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class K, class... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, int threads, size_t smem, cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int NT>
cudaError_t launch_lm_nt(const CUtensorMap& tw, const CUtensorMap& tx, const LmArgs& a, cudaStream_t st, bool pdl) {
  constexpr int kStage = kLmWBytes + 8 * NT * kLmK * 2;
  const size_t smem = (size_t)kLmRing * kStage + 2 * kLmRing * 8 + 1024;  // + alignment slack
  static DeviceOnce configured;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!configured.done(dev)) {
    e = cudaFuncSetAttribute(lm_head_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured.mark(dev);
  }
  return launch_pdl(lm_head_kernel<NT>, dim3((unsigned)(a.vocab / kLmRows)), kLmThreads, smem, st, pdl, tw, tx, a);
}

}  // namespace

cudaError_t launch_embed(const int* tokens, const uint16_t* table, int vocab, int H, int batch, uint16_t* x,
                         int* err, cudaStream_t st, bool pdl) {
  return launch_pdl(embed_kernel, dim3((unsigned)batch), 256, 0, st, pdl, tokens,
                    reinterpret_cast<const __nv_bfloat16*>(table), vocab, H, reinterpret_cast<__nv_bfloat16*>(x),
                    err);
}

cudaError_t launch_final_norm(const uint16_t* y, const float* g, int H, float eps, int batch, uint16_t* xg, float* r,
                              cudaStream_t st, bool pdl) {
  return launch_pdl(final_norm_kernel, dim3((unsigned)batch), 256, 0, st, pdl,
                    reinterpret_cast<const __nv_bfloat16*>(y), g, H, eps, reinterpret_cast<__nv_bfloat16*>(xg), r);
}

// Activation tiles of a tensor-core projection: the same 64-input x rows
// boxes (128-byte swizzle) as the LM head's activation; rows past `rows`
// read as zero.
bool make_act_tile_map(CUtensorMap* m, const void* x, int rows, int K) {
  return make_map(m, x, (uint64_t)K, (uint64_t)rows, 32);
}

// Activation tiles of an mma.sync projection: boxes of 136 inputs x box_rows
// rows, no swizzle, landing as rows of 272 bytes (128 inputs + 8 padding
// elements that the consumer never reads); rows past `rows` and inputs past K
// read as zero.
bool make_proj_tile_map(CUtensorMap* m, const void* x, int rows, int K, int box_rows) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {136, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_lm_head(const uint16_t* xg, const uint16_t* w, int vocab, int H, int batch, const float* r,
                           float* logits, int* err, cudaStream_t st, bool pdl) {
  const int nt = (batch + 7) / 8;
  CUtensorMap tw, tx;
  if (!make_map(&tw, w, (uint64_t)H, (uint64_t)vocab, kLmRows)) return cudaErrorInvalidValue;
  if (!make_map(&tx, xg, (uint64_t)H, (uint64_t)batch, (uint32_t)(8 * nt))) return cudaErrorInvalidValue;
  LmArgs a{r, logits, vocab, H, batch, err};
  switch (nt) {
    case 1: return launch_lm_nt<1>(tw, tx, a, st, pdl);
    case 2: return launch_lm_nt<2>(tw, tx, a, st, pdl);
    case 3: return launch_lm_nt<3>(tw, tx, a, st, pdl);
    default: return launch_lm_nt<4>(tw, tx, a, st, pdl);
  }
}

}  // namespace futr
