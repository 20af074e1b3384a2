// Offline weight packer and its canonical unpacker.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract: the fixed RMSNorm gain is folded into the weights and the
// decode projections use INT4 round-to-nearest weights laid out so that
// dequantization feeds MMA operands directly (explainer "FP8 Prefill + INT4
// Decode", section "INT4 Decode: letting dequantization feed directly into MMA
// operands").  Here the fragment is the sm_80+ mma.m16n8k16 A operand.
#include "futr_internal.cuh"

namespace futr {

namespace {

constexpr int kPackThreads = 128;
constexpr int kTileLd = kGroup + 1;  // padded fp32 row of the staged tile
constexpr int kCodeLd = kGroup + 4;  // padded int8 row of the staged codes

struct PackArgs {
  const float* src[3];   // row sources (QKV: wq, wk, wv; GU: gate, up; else [0])
  int split1, split2;    // QKV: q_rows, q_rows + kv_rows
  const float* gain;     // nullptr: no gain
  int kind;              // 0 QKV, 1 plain, 2 gate/up interleave
  int K, n_groups;
  uint8_t* out;          // section base
};

__device__ __forceinline__ const float* pack_row(const PackArgs& a, int R) {
  if (a.kind == 0) {
    if (R < a.split1) return a.src[0] + (size_t)R * a.K;
    if (R < a.split2) return a.src[1] + (size_t)(R - a.split1) * a.K;
    return a.src[2] + (size_t)(R - a.split2) * a.K;
  }
  if (a.kind == 2) {
    const int rb = R >> 7, lr = R & 127;
    const int j = 64 * rb + (lr & 63);
    return (lr < 64 ? a.src[0] : a.src[1]) + (size_t)j * a.K;
  }
  return a.src[0] + (size_t)R * a.K;
}

__global__ void __launch_bounds__(kPackThreads) pack_kernel(const PackArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* tile = reinterpret_cast<float*>(smem);                       // [128][129]
  int8_t* codes = reinterpret_cast<int8_t*>(smem + kRowsPerBlock * kTileLd * 4);  // [128][132]
  const int rb = blockIdx.x / a.n_groups, grp = blockIdx.x % a.n_groups;
  const int tid = threadIdx.x;
  const int c0 = grp * kGroup;

  // W' = W diag(g), one fp32 rounding, staged row by row (coalesced).
  for (int e = tid; e < kRowsPerBlock * kGroup; e += kPackThreads) {
    const int r = e >> 7, c = e & 127;
    float w = pack_row(a, rb * kRowsPerBlock + r)[c0 + c];
    if (a.gain) w = __fmul_rn(w, a.gain[c0 + c]);
    tile[r * kTileLd + c] = w;
  }
  __syncthreads();

  // One thread per output row: group absmax, fp16 scale, INT4 codes.
  {
    const int r = tid;
    float m = 0.f;
    for (int c = 0; c < kGroup; ++c) m = fmaxf(m, fabsf(tile[r * kTileLd + c]));
    const __half s = __float2half_rn(fminf(__fdiv_rn(m, 7.0f), 65504.0f));
    const float sf = __half2float(s);
    for (int c = 0; c < kGroup; ++c) {
      int q = 0;
      if (sf > 0.f) {
        q = __float2int_rn(__fdiv_rn(tile[r * kTileLd + c], sf));
        q = q < -8 ? -8 : (q > 7 ? 7 : q);
      }
      codes[r * kCodeLd + c] = (int8_t)q;
    }
    uint8_t* unit = a.out + ((size_t)rb * a.n_groups + grp) * kUnitBytes;
    reinterpret_cast<__half*>(unit + kUnitCodeBytes)[r] = s;
  }
  __syncthreads();

  // Fragment-ordered words: w = rt*256 + half*128 + lane*4 + j.
  uint32_t* unit_w = reinterpret_cast<uint32_t*>(a.out + ((size_t)rb * a.n_groups + grp) * kUnitBytes);
  for (int w = tid; w < kUnitCodeBytes / 4; w += kPackThreads) {
    const int rt = w >> 8, half = (w >> 7) & 1, lane = (w >> 2) & 31, j = w & 3;
    const int ks = 4 * half + j, gr = lane >> 2, t = lane & 3;
    const int r0 = 16 * rt + gr, r1 = r0 + 8, c = 16 * ks + 2 * t;
    const int rr[8] = {r0, r1, r0, r1, r0, r1, r0, r1};
    const int cc[8] = {c, c, c + 8, c + 8, c + 1, c + 1, c + 9, c + 9};
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= (uint32_t)((codes[rr[i] * kCodeLd + cc[i]] + 8) & 0xF) << (4 * i);
    unit_w[w] = word;
  }
}

__global__ void header_kernel(BlobHeader* dst, const BlobHeader h) { *dst = h; }

struct UnpackArgs {
  const uint8_t* sec;
  int rows, cols, n_groups;
  int map;  // 0 identity, 1 gate rows, 2 up rows
  int8_t* codes;
  uint16_t* scales;
};

__global__ void unpack_kernel(const UnpackArgs a) {
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (size_t)a.rows * a.cols) return;
  const int R = (int)(e / a.cols), C = (int)(e % a.cols);
  int SR = R;
  if (a.map == 1) SR = 128 * (R / 64) + (R % 64);
  if (a.map == 2) SR = 128 * (R / 64) + 64 + (R % 64);
  const int rb = SR >> 7, lr = SR & 127, rt = lr >> 4, rr = lr & 15, gr = rr & 7, upper = rr >> 3;
  const int grp = C >> 7, cc = C & 127, ks = cc >> 4, kk = cc & 15;
  const int t = (kk & 7) >> 1, odd = kk & 1, hi8 = kk >> 3;
  const int slot = upper + 2 * hi8 + 4 * odd;
  const int half = ks >> 2, j = ks & 3, lane = 4 * gr + t;
  const uint8_t* unit = a.sec + ((size_t)rb * a.n_groups + grp) * kUnitBytes;
  const uint32_t word = reinterpret_cast<const uint32_t*>(unit)[rt * 256 + half * 128 + lane * 4 + j];
  a.codes[e] = (int8_t)((int)((word >> (4 * slot)) & 0xF) - 8);
  if (cc == 0) a.scales[(size_t)R * a.n_groups + grp] = reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes)[lr];
}

}  // namespace

cudaError_t launch_pack(const futr_shape& s, const float* wq, const float* wk, const float* wv,
                        const float* wo, const float* wg, const float* wu, const float* wd,
                        const float* ga, const float* gm, uint8_t* blob, cudaStream_t st) {
  const BlobSections sec = blob_sections(s);
  const size_t smem = (size_t)kRowsPerBlock * kTileLd * 4 + kRowsPerBlock * kCodeLd;
  cudaError_t e = cudaFuncSetAttribute(pack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int q_rows = s.n_q_heads * s.head_dim, kv_rows = s.n_kv_heads * s.head_dim;
  for (int i = 0; i < 4; ++i) {
    PackArgs a{};
    a.K = sec.cols[i];
    a.n_groups = sec.cols[i] / kGroup;
    a.out = blob + sec.off[i];
    if (i == 0) {
      a.kind = 0; a.src[0] = wq; a.src[1] = wk; a.src[2] = wv; a.split1 = q_rows; a.split2 = q_rows + kv_rows;
      a.gain = ga;
    } else if (i == 1) {
      a.kind = 1; a.src[0] = wo; a.gain = nullptr;
    } else if (i == 2) {
      a.kind = 2; a.src[0] = wg; a.src[1] = wu; a.gain = gm;
    } else {
      a.kind = 1; a.src[0] = wd; a.gain = nullptr;
    }
    const int units = (sec.rows[i] / kRowsPerBlock) * a.n_groups;
    pack_kernel<<<units, kPackThreads, smem, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  BlobHeader h{};
  h.magic = kBlobMagic;
  h.version = 1;
  h.shape = s;
  header_kernel<<<1, 1, 0, st>>>(reinterpret_cast<BlobHeader*>(blob), h);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const futr_shape& s, const uint8_t* blob, int which, int8_t* codes,
                          uint16_t* scales, cudaStream_t st) {
  const BlobSections sec = blob_sections(s);
  UnpackArgs a{};
  int section = 0;
  switch (which) {
    case FUTR_PROJ_QKV: section = 0; a.map = 0; a.rows = sec.rows[0]; break;
    case FUTR_PROJ_O: section = 1; a.map = 0; a.rows = sec.rows[1]; break;
    case FUTR_PROJ_GATE: section = 2; a.map = 1; a.rows = s.inter; break;
    case FUTR_PROJ_UP: section = 2; a.map = 2; a.rows = s.inter; break;
    default: section = 3; a.map = 0; a.rows = sec.rows[3]; break;
  }
  a.sec = blob + sec.off[section];
  a.cols = sec.cols[section];
  a.n_groups = a.cols / kGroup;
  a.codes = codes;
  a.scales = scales;
  const size_t n = (size_t)a.rows * a.cols;
  unpack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace futr
