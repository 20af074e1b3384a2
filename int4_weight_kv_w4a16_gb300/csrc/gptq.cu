// GPTQ variant of the offline packer: the same INT4 blob (codes in [-8, 7],
// one fp16 scale per output row per 128 inputs, A-fragment order), with the
// codes chosen by GPTQ from each projection input's Hessian.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract, and the explainer's section "Accuracy cost: perplexity
// from 6.24 to 7.23": GPTQ codes in the round-to-nearest format, chosen with
// calibration data and approximate second-order information.  The steps are
// those of the published GPTQ algorithm (Frantar et al., 2022), in natural
// column order, without activation reordering:
//   H' = H with every dead input (H_jj = 0) given H_jj = 1 (its weight column
//        set to 0), plus damp * mean(diag H') on the diagonal;
//   U  = the upper Cholesky factor of H'^-1 (H'^-1 = U^T U);
//   columns j = 0..K-1 in order, on a float64 working copy W of W diag(g):
//   at the first column of a 128-input group its scales are fp16(max|fp32 w| /
//   7); c_j = clamp(rint(fp32(w_j) / s), -8, 7); e = (w_j - c_j s) / U_jj; the
//   columns not yet quantized take W[:, j+1:] -= e U[j, j+1:].
// All of it in float64 on the device:
//   U: with J the order-reversing permutation, J H' J = L L^T (lower Cholesky)
//      gives H' = (J L J)(J L J)^T with J L J upper triangular, so
//      U = (J L J)^-1 = J L^-1 J: a blocked Cholesky, then L^-1 by blocked
//      forward substitution, then the reversal;
//   the column sweep in blocks of 128 columns (one scale group): inside a
//      block the columns go one by one (one CTA per 32 rows, the block in
//      shared memory); the rest of the row takes the block's errors at once
//      (W[:, j1:] -= E U[block, j1:], a GEMM).
// Mathematically this is the column-by-column sweep; the order of the float64
// additions differs.
#include <cmath>

#include "futr_internal.cuh"

namespace futr {

namespace {

constexpr int kCB = 32;     // Cholesky / inverse block
constexpr int kGT = 64;     // GEMM tile (rows and columns)
constexpr int kGK = 16;     // GEMM k-chunk
constexpr int kSweepRows = 32;

// C[m][n] = beta * C[m][n] + alpha * sum_k A[m][k] * B[k][n] over m < M,
// n < N; B[k][n] = Bt ? B[n * ldb + k] : B[k * ldb + n].  lower: only tiles
// that reach the lower triangle (n <= m) are written, and only their n <= m
// entries.  Row-major fp64, 256 threads, 64 x 64 tiles.
struct GemmArgs {
  const double* A;
  const double* B;
  double* C;
  long long lda, ldb, ldc;
  int M, N, K;
  double alpha, beta;
  int Bt, lower;
};

__global__ void __launch_bounds__(256) gemm_f64_kernel(const GemmArgs g) {
  __shared__ double As[kGK][kGT + 1];
  __shared__ double Bs[kGK][kGT + 1];
  const int m0 = blockIdx.y * kGT, n0 = blockIdx.x * kGT;
  if (g.lower && n0 > m0 + kGT - 1) return;
  const int tid = threadIdx.x, tm = tid / 16, tn = tid % 16;
  double acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += kGK) {
    for (int e = tid; e < kGK * kGT; e += 256) {
      const int kk = e % kGK, mm = e / kGK;
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < g.M && k < g.K) ? g.A[m * g.lda + k] : 0.0;
    }
    for (int e = tid; e < kGK * kGT; e += 256) {
      int kk, nn;
      if (g.Bt) {
        kk = e % kGK;
        nn = e / kGK;
      } else {
        nn = e % kGT;
        kk = e / kGT;
      }
      const int n = n0 + nn, k = k0 + kk;
      double v = 0.0;
      if (n < g.N && k < g.K) v = g.Bt ? g.B[n * g.ldb + k] : g.B[k * g.ldb + n];
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kGK; ++kk) {
      double a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tm + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tn + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + tm + 16 * i, n = n0 + tn + 16 * j;
      if (m < g.M && n < g.N && (!g.lower || n <= m)) {
        double* c = g.C + m * g.ldc + n;
        *c = (g.beta == 0.0 ? 0.0 : g.beta * *c) + g.alpha * acc[i][j];
      }
    }
}

cudaError_t gemm(const GemmArgs& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  dim3 grid((unsigned)((g.N + kGT - 1) / kGT), (unsigned)((g.M + kGT - 1) / kGT));
  gemm_f64_kernel<<<grid, 256, 0, st>>>(g);
  return cudaGetLastError();
}

// diag[j] = H_jj with dead inputs (H_jj = 0) given 1; dead[j] flags them;
// shift[0] = damp * mean(diag) (one CTA, fixed summation order).
__global__ void __launch_bounds__(256) hess_diag_kernel(const double* H, int K, double damp, int* dead,
                                                         double* shift) {
  __shared__ double part[256];
  double s = 0.0;
  for (int j = threadIdx.x; j < K; j += 256) {
    const double h = H[(long long)j * K + j];
    dead[j] = h == 0.0;
    s += h == 0.0 ? 1.0 : h;
  }
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) shift[0] = damp * (part[0] / K);
}

// A = J H' J: A[i][j] = H'[K-1-i][K-1-j] (dead diagonal 1, dampened diagonal).
__global__ void hess_reverse_kernel(const double* H, int K, const int* dead, const double* shift, double* A) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)K * K) return;
  const int i = (int)(e / K), j = (int)(e % K);
  const int si = K - 1 - i, sj = K - 1 - j;
  double v = H[(long long)si * K + sj];
  if (si == sj) v = (dead[si] ? 1.0 : v) + shift[0];
  A[e] = v;
}

// Unblocked Cholesky of the kCB x kCB diagonal block at (k0, k0) of A (lower,
// in place); a pivot that is not positive sets *bad.
__global__ void __launch_bounds__(kCB * kCB) chol_diag_kernel(double* A, long long lda, int k0, int nb,
                                                              int* bad) {
  __shared__ double L[kCB][kCB + 1];
  const int r = threadIdx.x / kCB, c = threadIdx.x % kCB;
  L[r][c] = (r < nb && c < nb) ? A[(k0 + r) * lda + k0 + c] : 0.0;
  __syncthreads();
  for (int j = 0; j < nb; ++j) {
    if (r == j && c == j) {
      const double d = L[j][j];
      if (!(d > 0.0)) *bad = 1;
      L[j][j] = d > 0.0 ? sqrt(d) : 1.0;
    }
    __syncthreads();
    if (c == j && r > j) L[r][j] /= L[j][j];
    __syncthreads();
    if (r > j && c > j && c <= r) L[r][c] -= L[r][j] * L[c][j];
    __syncthreads();
  }
  if (r < nb && c < nb && c <= r) A[(k0 + r) * lda + k0 + c] = L[r][c];
}

// Rows i >= k0 + nb of the panel: A[i][k0:k0+nb] <- A[i][k0:k0+nb] L_kk^-T.
__global__ void __launch_bounds__(128) chol_panel_kernel(double* A, long long lda, int k0, int nb, int K) {
  __shared__ double L[kCB][kCB + 1];
  for (int e = threadIdx.x; e < kCB * kCB; e += 128) {
    const int r = e / kCB, c = e % kCB;
    L[r][c] = (r < nb && c <= r) ? A[(k0 + r) * lda + k0 + c] : 0.0;
  }
  __syncthreads();
  const int i = k0 + nb + blockIdx.x * 128 + threadIdx.x;
  if (i >= K) return;
  double x[kCB];
  double* row = A + i * lda + k0;
#pragma unroll
  for (int j = 0; j < kCB; ++j) {
    if (j < nb) {
      double v = row[j];
      for (int p = 0; p < j; ++p) v -= x[p] * L[j][p];
      x[j] = v / L[j][j];
    }
  }
#pragma unroll
  for (int j = 0; j < kCB; ++j)
    if (j < nb) row[j] = x[j];
}

// Block row [i0, i0 + nb) of X = L^-1 (X zero above the diagonal):
// X[i0.., 0:i0] = -inv(L_ii) T (T = L[i0.., 0:i0] X[0:i0, 0:i0], computed
// before), X[i0.., i0..] = inv(L_ii).  Each CTA inverts the small triangle
// itself and handles 64 columns.
__global__ void __launch_bounds__(128) tri_block_kernel(const double* Lm, long long ld, int i0, int nb,
                                                        const double* T, long long ldt, double* X) {
  __shared__ double Li[kCB][kCB + 1];
  __shared__ double Ld[kCB][kCB + 1];
  for (int e = threadIdx.x; e < kCB * kCB; e += 128) {
    const int r = e / kCB, c = e % kCB;
    Ld[r][c] = (r < nb && c <= r) ? Lm[(i0 + r) * ld + i0 + c] : 0.0;
    Li[r][c] = 0.0;
  }
  __syncthreads();
  // inverse of the lower triangle, one column per thread (forward substitution)
  if (threadIdx.x < nb) {
    const int c = threadIdx.x;
    for (int r = c; r < nb; ++r) {
      double v = r == c ? 1.0 : 0.0;
      for (int p = c; p < r; ++p) v -= Ld[r][p] * Li[p][c];
      Li[r][c] = v / Ld[r][r];
    }
  }
  __syncthreads();
  const int c0 = blockIdx.x * 64;
  for (int e = threadIdx.x; e < nb * 64; e += 128) {
    const int r = e / 64, cc = c0 + e % 64;
    if (cc < i0) {
      double v = 0.0;
      for (int p = 0; p <= r; ++p) v += Li[r][p] * T[p * ldt + cc];
      X[(i0 + r) * ld + cc] = -v;
    } else if (cc < i0 + nb) {
      X[(i0 + r) * ld + cc] = Li[r][cc - i0];
    }
  }
}

// U[i][j] = X[K-1-i][K-1-j] for j >= i (upper triangle of J X J), 0 below.
__global__ void reverse_upper_kernel(const double* X, int K, double* U) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)K * K) return;
  const int i = (int)(e / K), j = (int)(e % K);
  U[e] = j >= i ? X[(long long)(K - 1 - i) * K + (K - 1 - j)] : 0.0;
}

// The float64 working copy of one projection: W'[r][c] = fp32(W[r][c] g[c])
// (rows from up to three sources, QKV), 0 in dead input columns.
struct FoldArgs {
  const float* src[3];
  int split1, split2;
  const float* gain;
  const int* dead;
  int N, K;
  double* W;
};

__global__ void fold_kernel(const FoldArgs a) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)a.N * a.K) return;
  const int r = (int)(e / a.K), c = (int)(e % a.K);
  const float* row = r < a.split1 ? a.src[0] + (long long)r * a.K
                                   : (r < a.split2 ? a.src[1] + (long long)(r - a.split1) * a.K
                                                   : a.src[2] + (long long)(r - a.split2) * a.K);
  float w = row[c];
  if (a.gain) w = __fmul_rn(w, a.gain[c]);
  a.W[e] = a.dead[c] ? 0.0 : (double)w;
}

// One block of 128 columns [j0, j0 + 128) of the sweep, for 32 rows per CTA
// (4 threads a row, 32 columns each): the group's scales, then column by
// column its codes, its error e = (w - c s) / U_jj (into E) and the update of
// the block's later columns.  The block of U comes to shared memory.
__global__ void __launch_bounds__(128) sweep_block_kernel(double* W, long long ldw, int N, const double* U, int K,
                                                          int j0, double* E, int8_t* codes, __half* scales) {
  extern __shared__ double sm[];
  double* Ub = sm;                          // [128][128]
  double* Wb = sm + kGroup * kGroup;        // [32][128 + 1]
  const int tid = threadIdx.x, r = tid >> 2, part = tid & 3;
  const int row = blockIdx.x * kSweepRows + r;
  for (int e = tid; e < kGroup * kGroup; e += 128) {
    const int i = e / kGroup, j = e % kGroup;
    Ub[e] = U[(long long)(j0 + i) * K + j0 + j];
  }
  for (int e = tid; e < kSweepRows * kGroup; e += 128) {
    const int rr = e / kGroup, cc = e % kGroup;
    const int R = blockIdx.x * kSweepRows + rr;
    Wb[rr * (kGroup + 1) + cc] = R < N ? W[(long long)R * ldw + j0 + cc] : 0.0;
  }
  __syncthreads();
  double* w = Wb + r * (kGroup + 1);
  // the group's scale from its current weights: fp16(max |fp32 w| / 7)
  float m = 0.f;
  for (int cc = 32 * part; cc < 32 * part + 32; ++cc) m = fmaxf(m, fabsf((float)w[cc]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const __half s = __float2half_rn(fminf(__fdiv_rn(m, 7.0f), 65504.0f));
  const float sf = __half2float(s);
  const double sd = (double)sf;
  for (int j = 0; j < kGroup; ++j) {
    double e = 0.0;
    if (part == (j >> 5)) {
      const double wj = w[j];
      int c = 0;
      if (sf > 0.f) {
        c = __float2int_rn(__fdiv_rn((float)wj, sf));
        c = c < -8 ? -8 : (c > 7 ? 7 : c);
      }
      e = (wj - (double)c * sd) / Ub[j * kGroup + j];
      if (row < N) {
        codes[(long long)row * K + j0 + j] = (int8_t)c;
        E[(long long)row * kGroup + j] = e;
      }
    }
    e = __shfl_sync(0xffffffffu, e, (tid & ~3) | (j >> 5));
    for (int cc = max(j + 1, 32 * part); cc < 32 * part + 32; ++cc) w[cc] -= e * Ub[j * kGroup + cc];
    __syncwarp();
  }
  if (part == 0 && row < N) scales[(long long)row * (K / kGroup) + j0 / kGroup] = s;
}

// Blob section from canonical codes [rows][K] and scales [rows][K/128]:
// identity rows, or (gate/up) row block rb holding 64 rows of each matrix.
struct RepackArgs {
  const int8_t* codes[2];
  const __half* scales[2];
  int interleave, K, n_groups;
  uint8_t* out;
};

__global__ void __launch_bounds__(256) repack_kernel(const RepackArgs a) {
  const int rb = blockIdx.x / a.n_groups, grp = blockIdx.x % a.n_groups;
  auto src = [&](int lr, int& which) {
    if (!a.interleave) {
      which = 0;
      return rb * kRowsPerBlock + lr;
    }
    which = lr < 64 ? 0 : 1;
    return 64 * rb + (lr & 63);
  };
  uint8_t* unit = a.out + ((size_t)rb * a.n_groups + grp) * kUnitBytes;
  uint32_t* unit_w = reinterpret_cast<uint32_t*>(unit);
  for (int wi = threadIdx.x; wi < kUnitCodeBytes / 4; wi += 256) {
    const int rt = wi >> 8, half = (wi >> 7) & 1, lane = (wi >> 2) & 31, j = wi & 3;
    const int ks = 4 * half + j, gr = lane >> 2, t = lane & 3;
    const int r0 = 16 * rt + gr, c = grp * kGroup + 16 * ks + 2 * t;
    const int rr[8] = {r0, r0 + 8, r0, r0 + 8, r0, r0 + 8, r0, r0 + 8};
    const int cc[8] = {c, c, c + 8, c + 8, c + 1, c + 1, c + 9, c + 9};
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int which;
      const int R = src(rr[i], which);
      word |= (uint32_t)((a.codes[which][(long long)R * a.K + cc[i]] + 8) & 0xF) << (4 * i);
    }
    unit_w[wi] = word;
  }
  if (threadIdx.x < kRowsPerBlock) {
    int which;
    const int R = src(threadIdx.x, which);
    reinterpret_cast<__half*>(unit + kUnitCodeBytes)[threadIdx.x] = a.scales[which][(long long)R * a.n_groups + grp];
  }
}

__global__ void gptq_header_kernel(BlobHeader* dst, const BlobHeader h) { *dst = h; }

// Scratch layout of one packing (float64 K x K buffers for the Hessian's
// factor and inverse, the working weights, the block errors, the codes and
// scales of up to two matrices).
struct GptqScratch {
  size_t A, X, W, E, codes, scales, dead, shift, bad, total;
};

inline size_t al(size_t x) { return (x + 255) & ~size_t(255); }

GptqScratch gptq_layout(const futr_shape& s) {
  const BlobSections sec = blob_sections(s);
  size_t kmax = 0, nk = 0, nmax = 0, codes2 = 0, scales2 = 0;
  for (int i = 0; i < 4; ++i) {
    kmax = std::max(kmax, (size_t)sec.cols[i]);
    const size_t rows = i == 2 ? (size_t)s.inter : (size_t)sec.rows[i];  // gate and up one at a time
    nk = std::max(nk, rows * sec.cols[i]);
    nmax = std::max(nmax, rows);
    codes2 = std::max(codes2, (size_t)sec.rows[i] * sec.cols[i]);
    scales2 = std::max(scales2, (size_t)sec.rows[i] * (sec.cols[i] / kGroup));
  }
  GptqScratch L{};
  size_t off = 0;
  L.A = off; off = al(off + kmax * kmax * 8);
  L.X = off; off = al(off + kmax * kmax * 8);
  L.W = off; off = al(off + nk * 8);
  L.E = off; off = al(off + nmax * kGroup * 8);
  L.codes = off; off = al(off + codes2);
  L.scales = off; off = al(off + scales2 * 2);
  L.dead = off; off = al(off + kmax * 4);
  L.shift = off; off = al(off + 8);
  L.bad = off; off = al(off + 16);
  L.total = off;
  return L;
}

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(base) + off);
}

// U for Hessian H [K][K] into the scratch's A buffer (X used on the way).
cudaError_t factor(const double* H, int K, double damp, void* scr, const GptqScratch& L, cudaStream_t st) {
  double* A = at<double>(scr, L.A);
  double* X = at<double>(scr, L.X);
  int* dead = at<int>(scr, L.dead);
  double* shift = at<double>(scr, L.shift);
  int* bad = at<int>(scr, L.bad);
  const long long KK = (long long)K * K;
  const unsigned blocks = (unsigned)((KK + 255) / 256);
  hess_diag_kernel<<<1, 256, 0, st>>>(H, K, damp, dead, shift);
  hess_reverse_kernel<<<blocks, 256, 0, st>>>(H, K, dead, shift, A);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // lower Cholesky of A, blocked (right-looking)
  for (int k0 = 0; k0 < K; k0 += kCB) {
    const int nb = std::min(kCB, K - k0);
    chol_diag_kernel<<<1, kCB * kCB, 0, st>>>(A, K, k0, nb, bad);
    const int rest = K - k0 - nb;
    if (rest > 0) {
      chol_panel_kernel<<<(unsigned)((rest + 127) / 128), 128, 0, st>>>(A, K, k0, nb, K);
      GemmArgs g{};
      g.A = A + (long long)(k0 + nb) * K + k0;  // panel P [rest][nb]
      g.B = g.A;                                // P^T
      g.C = A + (long long)(k0 + nb) * K + k0 + nb;
      g.lda = g.ldb = g.ldc = K;
      g.M = g.N = rest;
      g.K = nb;
      g.alpha = -1.0;
      g.beta = 1.0;
      g.Bt = 1;
      g.lower = 1;
      e = gemm(g, st);
      if (e != cudaSuccess) return e;
    }
  }
  // X = L^-1 by block rows, each from T = L[i0.., 0:i0] X[0:i0, 0:i0]; T
  // (kCB x K doubles) lives in the working-weight buffer, unused until the sweep
  e = cudaMemsetAsync(X, 0, (size_t)KK * 8, st);
  if (e != cudaSuccess) return e;
  double* T = at<double>(scr, L.W);
  for (int i0 = 0; i0 < K; i0 += kCB) {
    const int nb = std::min(kCB, K - i0);
    if (i0 > 0) {
      GemmArgs g{};
      g.A = A + (long long)i0 * K;
      g.B = X;
      g.C = T;
      g.lda = g.ldb = K;
      g.ldc = K;
      g.M = nb;
      g.N = i0;
      g.K = i0;
      g.alpha = 1.0;
      g.beta = 0.0;
      e = gemm(g, st);
      if (e != cudaSuccess) return e;
    }
    tri_block_kernel<<<(unsigned)((i0 + nb + 63) / 64), 128, 0, st>>>(A, K, i0, nb, T, K, X);
  }
  reverse_upper_kernel<<<blocks, 256, 0, st>>>(X, K, A);
  return cudaGetLastError();
}

// The sweep of one matrix W [N][K] (already in the scratch's W buffer) under
// U (the A buffer): codes [N][K] and scales [N][K/128] into codes/scales.
cudaError_t sweep(int N, int K, void* scr, const GptqScratch& L, int8_t* codes, __half* scales, cudaStream_t st) {
  double* W = at<double>(scr, L.W);
  const double* U = at<double>(scr, L.A);
  double* E = at<double>(scr, L.E);
  const size_t smem = (size_t)(kGroup * kGroup + kSweepRows * (kGroup + 1)) * 8;
  cudaError_t e = cudaFuncSetAttribute(sweep_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  for (int j0 = 0; j0 < K; j0 += kGroup) {
    sweep_block_kernel<<<(unsigned)((N + kSweepRows - 1) / kSweepRows), 128, smem, st>>>(W, K, N, U, K, j0, E, codes,
                                                                                          scales);
    const int j1 = j0 + kGroup;
    if (j1 < K) {
      GemmArgs g{};
      g.A = E;
      g.B = U + (long long)j0 * K + j1;
      g.C = W + j1;
      g.lda = kGroup;
      g.ldb = K;
      g.ldc = K;
      g.M = N;
      g.N = K - j1;
      g.K = kGroup;
      g.alpha = -1.0;
      g.beta = 1.0;
      e = gemm(g, st);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaGetLastError();
}

cudaError_t fold(const FoldArgs& f, cudaStream_t st) {
  const long long n = (long long)f.N * f.K;
  fold_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(f);
  return cudaGetLastError();
}

}  // namespace

size_t gptq_scratch_bytes(const futr_shape& s) { return gptq_layout(s).total; }

cudaError_t launch_pack_gptq(const futr_shape& s, const float* wq, const float* wk, const float* wv,
                             const float* wo, const float* wg, const float* wu, const float* wd, const float* ga,
                             const float* gm, const double* h_attn, const double* h_o, const double* h_mlp,
                             const double* h_down, double damp, void* scratch, uint8_t* blob, int* bad_host,
                             cudaStream_t st) {
  const BlobSections sec = blob_sections(s);
  const GptqScratch L = gptq_layout(s);
  int8_t* codes = at<int8_t>(scratch, L.codes);
  __half* scales = at<__half>(scratch, L.scales);
  const int* dead = at<int>(scratch, L.dead);
  cudaError_t e = cudaMemsetAsync(at<int>(scratch, L.bad), 0, 4, st);
  if (e != cudaSuccess) return e;
  const int q_rows = s.n_q_heads * s.head_dim, kv_rows = s.n_kv_heads * s.head_dim;
  const int I = s.inter, H = s.hidden;
  auto one = [&](const float* const* src, int split1, int split2, const float* gain, int N, int K, int8_t* c,
                 __half* sc) -> cudaError_t {
    FoldArgs f{};
    for (int i = 0; i < 3; ++i) f.src[i] = src[i];
    f.split1 = split1;
    f.split2 = split2;
    f.gain = gain;
    f.dead = dead;
    f.N = N;
    f.K = K;
    f.W = at<double>(scratch, L.W);
    cudaError_t r = fold(f, st);
    if (r != cudaSuccess) return r;
    return sweep(N, K, scratch, L, c, sc, st);
  };
  auto repack = [&](int section, int interleave, const int8_t* c0, const __half* s0, const int8_t* c1,
                    const __half* s1) -> cudaError_t {
    RepackArgs r{};
    r.codes[0] = c0;
    r.codes[1] = c1;
    r.scales[0] = s0;
    r.scales[1] = s1;
    r.interleave = interleave;
    r.K = sec.cols[section];
    r.n_groups = sec.cols[section] / kGroup;
    r.out = blob + sec.off[section];
    repack_kernel<<<(unsigned)((sec.rows[section] / kRowsPerBlock) * r.n_groups), 256, 0, st>>>(r);
    return cudaGetLastError();
  };
  // QKV: one matrix (rows Wq; Wk; Wv) under the attention input's Hessian
  {
    const float* src[3] = {wq, wk, wv};
    if ((e = factor(h_attn, H, damp, scratch, L, st)) != cudaSuccess) return e;
    if ((e = one(src, q_rows, q_rows + kv_rows, ga, sec.rows[0], H, codes, scales)) != cudaSuccess) return e;
    if ((e = repack(0, 0, codes, scales, nullptr, nullptr)) != cudaSuccess) return e;
  }
  // O under the attention output's Hessian
  {
    const int K = s.n_q_heads * s.head_dim;
    const float* src[3] = {wo, wo, wo};
    if ((e = factor(h_o, K, damp, scratch, L, st)) != cudaSuccess) return e;
    if ((e = one(src, H, H, nullptr, H, K, codes, scales)) != cudaSuccess) return e;
    if ((e = repack(1, 0, codes, scales, nullptr, nullptr)) != cudaSuccess) return e;
  }
  // gate and up, each under the MLP input's Hessian (one factor for both)
  {
    const float* sg[3] = {wg, wg, wg};
    const float* su[3] = {wu, wu, wu};
    int8_t* cg = codes;
    int8_t* cu = codes + (size_t)I * H;
    __half* sgs = scales;
    __half* sus = scales + (size_t)I * (H / kGroup);
    if ((e = factor(h_mlp, H, damp, scratch, L, st)) != cudaSuccess) return e;
    if ((e = one(sg, I, I, gm, I, H, cg, sgs)) != cudaSuccess) return e;
    if ((e = one(su, I, I, gm, I, H, cu, sus)) != cudaSuccess) return e;
    if ((e = repack(2, 1, cg, sgs, cu, sus)) != cudaSuccess) return e;
  }
  // down under the SwiGLU output's Hessian
  {
    const float* src[3] = {wd, wd, wd};
    if ((e = factor(h_down, I, damp, scratch, L, st)) != cudaSuccess) return e;
    if ((e = one(src, H, H, nullptr, H, I, codes, scales)) != cudaSuccess) return e;
    if ((e = repack(3, 0, codes, scales, nullptr, nullptr)) != cudaSuccess) return e;
  }
  BlobHeader h{};
  h.magic = kBlobMagic;
  h.version = 1;
  h.shape = s;
  gptq_header_kernel<<<1, 1, 0, st>>>(reinterpret_cast<BlobHeader*>(blob), h);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaMemcpyAsync(bad_host, at<int>(scratch, L.bad), 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return e;
  return cudaStreamSynchronize(st);
}

}  // namespace futr
