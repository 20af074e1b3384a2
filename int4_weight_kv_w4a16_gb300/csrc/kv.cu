// INT4 KV-cache copy: RoPE table, bulk append (rotate + quantize), canonical
// read-back.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract: decode reads an INT4 copy of the KV cache, rotated
// block-diagonally with a Hadamard matrix so that outlier channels cost less
// quantization error, and keys are stored in the tensor cores' fragment layout.  Here keys are stored as the
// mma.m16n8k16 B operand of q.k (k = head dims, n = positions) and values as
// the B operand of p.V (k = positions, n = head dims).
#include "futr_internal.cuh"

namespace futr {

namespace {

__global__ void rope_table_kernel(float2* table, int cap, int d, double theta) {
  const int half = d / 2;
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (size_t)cap * half) return;
  const int p = (int)(e / half), i = (int)(e % half);
  const double inv = pow(theta, -2.0 * (double)i / (double)d);
  double sn, cs;
  sincos((double)p * inv, &sn, &cs);
  table[e] = make_float2((float)cs, (float)sn);
}

template <int J>
__global__ void __launch_bounds__(256) kv_append_kernel(KvView kv, int seq0, const int* pos, int n_tok,
                                                       const uint16_t* k, const uint16_t* v, int nh,
                                                       float c, int* err) {
  constexpr int d = 32 * J;
  __shared__ int8_t vcode[16][d];
  __shared__ __half vscale[16];
  __shared__ int8_t scratch[8][d];
  const int b = blockIdx.z, kvh = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p0 = pos[b];
  if (p0 < 0 || (long)p0 + n_tok > kv.cap) {
    if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0) set_err(err, FUTR_ERR_OUT_OF_RANGE);
    return;
  }
  const int tile = (p0 >> 4) + (int)blockIdx.x;
  const int lo = max(tile * 16, p0), hi = min(tile * 16 + 16, p0 + n_tok);
  if (lo >= hi) return;
  uint8_t* strm = kv.stream(seq0 + b, kvh);
  const size_t row0 = ((size_t)b * kv.n_kv + kvh) * n_tok;
  for (int p = lo + warp; p < hi; p += 8) {
    const size_t src = (row0 + (p - p0)) * d;
    float x[J];
    int code[J];
#pragma unroll
    for (int j = 0; j < J; ++j) x[j] = __uint_as_float((uint32_t)k[src + lane + 32 * j] << 16);
    warp_fwht<J>(x, nh, c);
    __half s = warp_quant<J>(x, code);
    store_k_token<J>(strm, kv.cap, p, code, s, scratch[warp]);
#pragma unroll
    for (int j = 0; j < J; ++j) x[j] = __uint_as_float((uint32_t)v[src + lane + 32 * j] << 16);
    warp_fwht<J>(x, nh, c);
    s = warp_quant<J>(x, code);
#pragma unroll
    for (int j = 0; j < J; ++j) vcode[p & 15][lane + 32 * j] = (int8_t)code[j];
    if (lane == 0) vscale[p & 15] = s;
  }
  __syncthreads();
  // Values: one thread per word of the 16-position tile; only nibbles of
  // positions in [lo, hi) change.
  uint32_t* vt = reinterpret_cast<uint32_t*>(strm + (size_t)kv.cap * (d / 2) + (size_t)tile * (8 * d));
  for (int w = threadIdx.x; w < 32 * (d / 16); w += blockDim.x) {
    const int ln = w / (d / 16), j = w % (d / 16), gr = ln >> 2, t = ln & 3;
    uint32_t word = vt[w];
    const int pp[8] = {2 * t, 2 * t + 8, 2 * t, 2 * t + 8, 2 * t + 1, 2 * t + 9, 2 * t + 1, 2 * t + 9};
    const int dd[8] = {16 * j + gr, 16 * j + gr, 16 * j + 8 + gr, 16 * j + 8 + gr,
                       16 * j + gr, 16 * j + gr, 16 * j + 8 + gr, 16 * j + 8 + gr};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int p = tile * 16 + pp[i];
      if (p >= lo && p < hi) {
        word = (word & ~(0xFu << (4 * i))) | ((uint32_t)((vcode[pp[i]][dd[i]] + 8) & 0xF) << (4 * i));
      }
    }
    vt[w] = word;
  }
  __half* vs = reinterpret_cast<__half*>(strm + (size_t)kv.cap * d + 2ull * kv.cap);
  if (threadIdx.x < 16) {
    const int p = tile * 16 + threadIdx.x;
    if (p >= lo && p < hi) vs[p] = vscale[threadIdx.x];
  }
}

__global__ void kv_read_kernel(KvView kv, int seq, int n_pos, int8_t* kc, uint16_t* ks, int8_t* vc,
                               uint16_t* vs) {
  const int p = blockIdx.x, h = blockIdx.y, dim = threadIdx.x, d = kv.d;
  const uint8_t* strm = kv.stream(seq, h);
  {  // key nibble
    const int j = dim / 32, u = dim % 32, half16 = u / 16, w16 = u % 16;
    const int hi8 = w16 / 8, odd = w16 & 1, t = (w16 % 8) / 2;
    const int slot = hi8 + 2 * half16 + 4 * odd, lane = 4 * (p & 7) + t;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(strm + (size_t)(p >> 3) * (4 * d) + lane * (d / 8) + 4 * j);
    kc[((size_t)h * n_pos + p) * d + dim] = (int8_t)((int)((w >> (4 * slot)) & 0xF) - 8);
  }
  {  // value nibble
    const int p16 = p & 15, t = (p16 & 7) >> 1, hi = p16 >> 3, odd = p16 & 1;
    const int j = dim / 16, r = dim % 16, gr = r % 8, upper8 = r / 8;
    const int slot = hi + 2 * upper8 + 4 * odd, lane = 4 * gr + t;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(strm + (size_t)kv.cap * (d / 2) +
                                                          (size_t)(p >> 4) * (8 * d) + lane * (d / 4) + 4 * j);
    vc[((size_t)h * n_pos + p) * d + dim] = (int8_t)((int)((w >> (4 * slot)) & 0xF) - 8);
  }
  if (dim == 0) {
    ks[(size_t)h * n_pos + p] = reinterpret_cast<const uint16_t*>(strm + (size_t)kv.cap * d)[p];
    vs[(size_t)h * n_pos + p] = reinterpret_cast<const uint16_t*>(strm + (size_t)kv.cap * d + 2ull * kv.cap)[p];
  }
}

KvView layer_view(const futr_kv& kv, int layer) {
  KvView v;
  v.base = reinterpret_cast<uint8_t*>(kv.base) +
           (uint64_t)layer * kv.max_batch * kv.shape.n_kv_heads * kv.stream_bytes;
  v.stream_bytes = kv.stream_bytes;
  v.cap = kv.capacity;
  v.d = kv.shape.head_dim;
  v.n_kv = kv.shape.n_kv_heads;
  return v;
}

}  // namespace

KvView kv_layer_view(const futr_kv& kv, int layer) { return layer_view(kv, layer); }

cudaError_t launch_rope_table(float2* table, int cap, int d, float theta, cudaStream_t st) {
  const size_t n = (size_t)cap * (d / 2);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(table, cap, d, (double)theta);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const futr_kv& kv, int layer, int seq0, int batch, const int* pos, int n_tok,
                             const uint16_t* k, const uint16_t* v, int* err, cudaStream_t st) {
  const KvView view = layer_view(kv, layer);
  const int nh = kv.shape.had_block;
  const float c = (float)(1.0 / sqrt((double)nh));
  dim3 grid((unsigned)((n_tok + 15) / 16 + 1), (unsigned)kv.shape.n_kv_heads, (unsigned)batch);
  if (kv.shape.head_dim == 128)
    kv_append_kernel<4><<<grid, 256, 0, st>>>(view, seq0, pos, n_tok, k, v, nh, c, err);
  else
    kv_append_kernel<2><<<grid, 256, 0, st>>>(view, seq0, pos, n_tok, k, v, nh, c, err);
  return cudaGetLastError();
}

cudaError_t launch_kv_read(const futr_kv& kv, int layer, int seq, int n_pos, int8_t* kc, uint16_t* ks,
                           int8_t* vc, uint16_t* vs, cudaStream_t st) {
  const KvView view = layer_view(kv, layer);
  dim3 grid((unsigned)n_pos, (unsigned)kv.shape.n_kv_heads);
  kv_read_kernel<<<grid, kv.shape.head_dim, 0, st>>>(view, seq, n_pos, kc, ks, vc, vs);
  return cudaGetLastError();
}

}  // namespace futr
