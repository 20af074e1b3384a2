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
//   warp 4 (producer): per 128-input group, one ring stage of shared memory
//     receives by 1-D bulk copies (mbarrier completion) the weight unit (codes
//     + scales, 8448 B) and the matching activation tile (one 256-byte row per
//     batch row, rows padded to 272 B).  Weight units of the first stages are
//     issued before griddepcontrol.wait, so weight streaming overlaps the
//     previous kernel; activation tiles follow the wait.
//   warps 0..3 (consumers): warp w owns rows 32w..32w+31 (two 16-row MMA
//     tiles sharing each B fragment); per group it reads its 64 bytes of
//     nibbles and four scales, builds the B fragments with ldmatrix from the
//     stage's tile, issues 2*8*NT mma, squares its share of the tile for the
//     RMSNorm sum of squares and releases the stage.
//   split-K: each CTA writes a partial [batch][128] (+ that sum of squares);
//     the last CTA of a row block (arrival counter, no spinning) adds the
//     partials in fixed order and runs the epilogue:
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

constexpr int kCW = 4;                    // consumer warps
constexpr int kMT = 2;                    // 16-row MMA tiles per consumer warp
constexpr int kThreads = (kCW + 1) * 32;  // + producer warp
constexpr int kRecCols = kRowsPerBlock / 4 + 1;  // float4 columns per batch row of a split record
constexpr int kRecLd = 4 * kRecCols;             // floats per batch row of a split record
static_assert(kCW * 32 == kRowsPerBlock, "one consumer thread per output row");

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
}

// Position and RoPE (cos, sin) of one head task: cs[j] pairs dims lane + 32 j
// and lane + 32 j + d/2.
struct HeadPre {
  int p;
  float2 cs[2];
};

// The head tasks' positions and RoPE factors in shared memory, loaded by many
// threads at once ahead of the epilogue: hcs[(task * 2 + j) * 32 + lane],
// hpos[task].  Item i = (task, lane) for i = first, first + stride, ...
__device__ __forceinline__ void fill_head_cache(const ProjArgs& a, int rb, float2* hcs, int* hpos, int first,
                                                int stride) {
  const int hpr = kRowsPerBlock / a.d, total = a.batch * hpr * 32, half = a.d / 2;
  // four items per round: their position loads, then their table loads, are
  // in flight together
  for (int i0 = first; i0 < total; i0 += 4 * stride) {
    int p[4];
    float2 c0[4], c1[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * stride;
      p[u] = i < total ? a.pos[(i >> 5) / hpr] : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * stride, task = i >> 5, l = i & 31;
      c0[u] = c1[u] = make_float2(1.f, 0.f);
      if (i < total && rb * hpr + task % hpr < a.Hq + a.Hkv) {  // q and k heads are rotated by position
        const int pp = p[u] >= 0 && p[u] < a.kv.cap ? p[u] : 0;
        c0[u] = a.rope[(size_t)pp * half + l];
        if (half > 32) c1[u] = a.rope[(size_t)pp * half + l + 32];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * stride, task = i >> 5, l = i & 31;
      if (i < total) {
        hcs[(task * 2) * 32 + l] = c0[u];
        hcs[(task * 2 + 1) * 32 + l] = c1[u];
        if (l == 0) hpos[task] = p[u];
      }
    }
  }
}

template <int J>
__device__ void qkv_head_epilogue(const ProjArgs& a, const float* red, int n, int hl, int hg, float r,
                                  const HeadPre& pre) {
  constexpr int d = 32 * J;
  const int lane = threadIdx.x & 31;
  float v[J];
#pragma unroll
  for (int j = 0; j < J; ++j) v[j] = red[n * kRedLd + hl * d + lane + 32 * j] * r;
  const int p = pre.p;
  const bool is_q = hg < a.Hq, is_k = !is_q && hg < a.Hq + a.Hkv;
  const bool p_ok = p >= 0 && p < a.kv.cap;
  if (is_q || is_k) {
    // rotate-half RoPE: dims i and i + d/2 (lane-local: element j pairs j + J/2)
#pragma unroll
    for (int j = 0; j < J / 2; ++j) {
      const float2 cs = pre.cs[j];
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

// Activation tile of group g into a ring stage: one 256-byte bulk copy per
// batch row, rows kTileLd elements apart.
__device__ __forceinline__ void issue_tile(const ProjArgs& a, uint8_t* stage, int g, uint64_t* bar) {
  uint8_t* dst = stage + kUnitBytes;
  const __nv_bfloat16* src = a.xin + (size_t)g * kGroup;
  for (int n = 0; n < a.batch; ++n) bulk_g2s(dst + n * (kTileLd * 2), src + (size_t)n * a.K, kGroup * 2, bar);
}

template <int NT, int EPI>
__device__ __forceinline__ void proj_body(const ProjArgs& a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.x / a.S, sk = blockIdx.x - rb * a.S;
  const int g0 = (int)(((long long)sk * a.n_groups) / a.S);
  const int g1 = (int)(((long long)(sk + 1) * a.n_groups) / a.S);
  const int ng = g1 - g0, R = a.ring;

  uint8_t* stages = smem;
  float* ss = reinterpret_cast<float*>(smem + a.off_misc);  // [32] sum of squares per batch row
  int* flag = reinterpret_cast<int*>(ss + 32);                // [4]
  uint64_t* full = reinterpret_cast<uint64_t*>(flag + 4);
  uint64_t* empty = full + kMaxRing;
  float* red = reinterpret_cast<float*>(smem);  // epilogue [NT*8][kRedLd], aliases the stages

  if (tid == 0) {
    flag[0] = 0;
    flag[1] = 0;
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();

  const uint8_t* unit0 = a.w + ((size_t)rb * a.n_groups + g0) * kUnitBytes;
  if (warp == kCW) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const uint32_t tx = kUnitBytes + (uint32_t)a.batch * kGroup * 2;
      const int pre = ng < R ? ng : R;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], tx);
        bulk_g2s(stages + (size_t)i * a.stage_bytes, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[i]);
      }
      pdl_wait();  // the activations come from the previous kernel
      const unsigned long long deadline = global_ns() + kWaitNs;
      for (int i = 0; i < pre; ++i) issue_tile(a, stages + (size_t)i * a.stage_bytes, g0 + i, &full[i]);
      int slot = 0;
      uint32_t phase = 0;
      for (int i = R; i < ng; ++i) {
        if (!mbar_wait_until(&empty[slot], phase, deadline)) {
          set_err(a.err, FUTR_ERR_TIMEOUT);
          break;
        }
        uint8_t* st = stages + (size_t)slot * a.stage_bytes;
        mbar_arrive_expect_tx(&full[slot], tx);
        bulk_g2s(st, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[slot]);
        issue_tile(a, st, g0 + i, &full[slot]);
        if (++slot == R) {
          slot = 0;
          phase ^= 1u;
        }
      }
    } else {
      pdl_wait();
    }
    return;
  }

  // ----------------------------------------------------------- consumers --
  pdl_wait();
  const unsigned long long deadline = global_ns() + kWaitNs;
  bool ok = true;

  float acc[kMT][NT][4];
#pragma unroll
  for (int m = 0; m < kMT; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][nt][e] = 0.f;

  const int gr = lane >> 2;
  // ldmatrix row offsets (elements, within a stage's tile) of this lane: batch
  // row 8nt + (lane & 7), column block (lane >> 3).  Rows past the batch read
  // row 0 instead: they only feed MMA columns that are never stored.
  int xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = 8 * nt + (lane & 7);
    xrow[nt] = (n < a.batch ? n : 0) * kTileLd + 8 * (lane >> 3);
  }
  // RMSNorm sum of squares of the activations: per group, consumer thread t
  // squares the 8 elements of tile row t / 16 + 8p, columns 8 (t % 16) .. +7
  // (16 lanes of one warp cover a row)
  const int sq_off = (tid >> 4) * kTileLd + 8 * (tid & 15);
  float ssq[NT];
#pragma unroll
  for (int p = 0; p < NT; ++p) ssq[p] = 0.f;
  int slot = 0;
  uint32_t phase = 0;
  for (int i = 0; i < ng; ++i) {
    if (!mbar_wait_until(&full[slot], phase, deadline)) {
      ok = false;
      break;
    }
    const uint8_t* st = stages + (size_t)slot * a.stage_bytes;
    const __nv_bfloat16* tile = reinterpret_cast<const __nv_bfloat16*>(st + kUnitBytes);
    // this warp's row tiles kMT*warp .. +kMT-1: 1024 contiguous bytes each
    const uint4* wt = reinterpret_cast<const uint4*>(st + kMT * warp * 1024);
    uint32_t words[kMT][8];
    float s_lo[kMT], s_hi[kMT];
    const __half* sc = reinterpret_cast<const __half*>(st + kUnitCodeBytes);
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      const uint4 w0 = wt[64 * m + lane], w1 = wt[64 * m + 32 + lane];
      words[m][0] = w0.x; words[m][1] = w0.y; words[m][2] = w0.z; words[m][3] = w0.w;
      words[m][4] = w1.x; words[m][5] = w1.y; words[m][6] = w1.z; words[m][7] = w1.w;
      const int r0 = (kMT * warp + m) * 16 + gr;
      s_lo[m] = __half2float(sc[r0]);
      s_hi[m] = __half2float(sc[r0 + 8]);
    }

    float dpart[kMT][NT][4];
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dpart[m][nt][e] = 0.f;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      uint32_t bfr[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) ldmatrix_x4(bfr[nt], tile + xrow[nt] + 32 * kp);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          const uint32_t w = words[m][2 * kp + h];
          uint32_t af[4];
          nib4_bf16x2(w, af);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(dpart[m][nt], af, bfr[nt][2 * h], bfr[nt][2 * h + 1]);
        }
    }
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[m][nt][0] = fmaf(s_lo[m], dpart[m][nt][0], acc[m][nt][0]);
        acc[m][nt][1] = fmaf(s_lo[m], dpart[m][nt][1], acc[m][nt][1]);
        acc[m][nt][2] = fmaf(s_hi[m], dpart[m][nt][2], acc[m][nt][2]);
        acc[m][nt][3] = fmaf(s_hi[m], dpart[m][nt][3], acc[m][nt][3]);
      }
    if (EPI != kEpiResid) {
#pragma unroll
      for (int p = 0; p < NT; ++p)
        if ((tid >> 4) + 8 * p < a.batch) {
          const uint4 v = *reinterpret_cast<const uint4*>(tile + sq_off + 8 * p * kTileLd);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(u[j] << 16), hi = __uint_as_float(u[j] & 0xffff0000u);
            ssq[p] = fmaf(lo, lo, fmaf(hi, hi, ssq[p]));
          }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the stage
    if (++slot == R) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (EPI != kEpiResid) {
    // the 16 lanes of a half-warp hold the 16 column blocks of one row
#pragma unroll
    for (int p = 0; p < NT; ++p) {
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) ssq[p] += __shfl_xor_sync(0xffffffffu, ssq[p], o);
      const int n = (tid >> 4) + 8 * p;
      if ((tid & 15) == 0 && n < a.batch) ss[n] = ssq[p];
    }
  }
  // the residual rows of this block (RESID): with one batch tile loaded now,
  // overlapping the split handshake; with more, in one burst after the
  // reduction, which keeps them out of its registers
  constexpr bool kEarly = NT == 1;
  __nv_bfloat16 rres[EPI == kEpiResid ? NT * 8 : 1];
  auto load_resid = [&]() {
    if (EPI == kEpiResid) {
#pragma unroll
      for (int n = 0; n < NT * 8; ++n)
        rres[n] = n < a.batch ? a.resid[(size_t)n * a.out_ld + (size_t)rb * kRowsPerBlock + tid]
                              : __float2bfloat16_rn(0.f);
    }
  };
  if (kEarly) load_resid();
  // QKV: the head tasks' positions and RoPE factors go to shared memory after
  // the epilogue tile and the split-sum groups (the ring is free by then)
  float2* hcs = reinterpret_cast<float2*>(red + NT * 8 * kRedLd + 4 * kCW * 32);
  int* hpos = reinterpret_cast<int*>(hcs + a.batch * (kRowsPerBlock / a.d) * 64);
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
    for (int m = 0; m < kMT; ++m) {
      const int r0 = (kMT * warp + m) * 16 + gr;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int n0 = 8 * nt + 2 * t;
        red[n0 * kRedLd + r0] = acc[m][nt][0];
        red[(n0 + 1) * kRedLd + r0] = acc[m][nt][1];
        red[n0 * kRedLd + r0 + 8] = acc[m][nt][2];
        red[(n0 + 1) * kRedLd + r0 + 8] = acc[m][nt][3];
      }
    }
  }
  consumer_sync();

  if (a.S > 1) {
    // publish this split's partial record: per batch row 32 float4 of sums and
    // one float4 (sum of squares, 0, 0, 0); then count arrivals
    float* rec = a.part + ((size_t)rb * a.S + sk) * a.rec_floats;
    const int items = a.batch * kRecCols;
    for (int e = tid; e < items; e += kCW * 32) {
      const int n = e / kRecCols, c4 = e - kRecCols * n;
      const float4 v = c4 < 32 ? reinterpret_cast<const float4*>(red + n * kRedLd)[c4]
                               : make_float4(EPI != kEpiResid ? ss[n] : 0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4*>(rec + n * kRecLd)[c4] = v;
    }
    consumer_sync();
    if (tid == 0)
      flag[0] = atom_add_acq_rel_gpu(&a.cnt[rb], 1u) == (unsigned)(a.S - 1) ? 1 : 0;
    else if (EPI == kEpiQkv)
      fill_head_cache(a, rb, hcs, hpos, tid - 1, kCW * 32 - 1);  // overlaps the arrival
    consumer_sync();
    if (!flag[0]) return;
    // The last CTA adds the S records.  With few columns (small batch), G
    // groups of threads each add a contiguous range of splits, all loads of a
    // range in flight together; the G group sums are then added in group
    // order.  The order is fixed, so the result is deterministic.
    const int G = items >= kCW * 32 ? 1 : (kCW * 32) / items;
    float4* gsum = reinterpret_cast<float4*>(red + NT * 8 * kRedLd);  // [G][items], G > 1 only
    const float* part_rb = a.part + (size_t)rb * a.S * a.rec_floats;
    if (G == 1) {
      // Many columns (batch >= 4): thread t owns columns t + 128 j and adds
      // them split by split, the loads of all its columns for one split in
      // flight together (the sum of each column stays in split order).
      constexpr int kJ = (NT * 8 * kRecCols + kCW * 32 - 1) / (kCW * 32);
      float4 s4[kJ];
      int col[kJ];
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        s4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int e = tid + kCW * 32 * j;
        col[j] = e < items ? e : -1;  // float4 index n * kRecCols + c4 of the record
      }
      // kSP splits per round: their loads are in flight together, then added
      // in split order
      constexpr int kSP = NT == 1 ? 1 : 2;
      const float4* rec4 = reinterpret_cast<const float4*>(part_rb);
      const size_t step = a.rec_floats / 4;
      for (int s0 = 0; s0 < a.S; s0 += kSP) {
        float4 v[kSP][kJ];
#pragma unroll
        for (int q = 0; q < kSP; ++q)
#pragma unroll
          for (int j = 0; j < kJ; ++j)
            if (col[j] >= 0 && s0 + q < a.S) v[q][j] = __ldcg(rec4 + (size_t)(s0 + q) * step + col[j]);
#pragma unroll
        for (int q = 0; q < kSP; ++q)
#pragma unroll
          for (int j = 0; j < kJ; ++j)
            if (col[j] >= 0 && s0 + q < a.S) {
              s4[j].x += v[q][j].x; s4[j].y += v[q][j].y; s4[j].z += v[q][j].z; s4[j].w += v[q][j].w;
            }
      }
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        if (col[j] >= 0) {
          const int n = col[j] / kRecCols, c4 = col[j] - kRecCols * n;
          if (c4 < 32)
            reinterpret_cast<float4*>(red + n * kRedLd)[c4] = s4[j];
          else
            ss[n] = s4[j].x;
        }
    }
    for (int t = tid; G > 1 && t < G * items; t += kCW * 32) {
      const int grp = t / items, e = t - grp * items;
      const int n = e / kRecCols, c4 = e - kRecCols * n;
      const int s_lo = grp * a.S / G, s_hi = (grp + 1) * a.S / G;
      const float4* src = reinterpret_cast<const float4*>(part_rb + n * kRecLd) + c4;
      float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = s_lo; s0 < s_hi; s0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < s_hi) v[j] = __ldcg(src + (size_t)(s0 + j) * (a.rec_floats / 4));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < s_hi) {
            s4.x += v[j].x; s4.y += v[j].y; s4.z += v[j].z; s4.w += v[j].w;
          }
      }
      gsum[t] = s4;
    }
    if (G > 1) {
      consumer_sync();
      for (int e = tid; e < items; e += kCW * 32) {
        float4 s4 = gsum[e];
        for (int grp = 1; grp < G; ++grp) {
          const float4 v = gsum[grp * items + e];
          s4.x += v.x; s4.y += v.y; s4.z += v.z; s4.w += v.w;
        }
        const int n = e / kRecCols, c4 = e - kRecCols * n;
        if (c4 < 32)
          reinterpret_cast<float4*>(red + n * kRedLd)[c4] = s4;
        else
          ss[n] = s4.x;
      }
    }
    if (tid == 0) a.cnt[rb] = 0u;  // self-reset for the next launch
    consumer_sync();
  }

  if (!kEarly) load_resid();
  if (EPI == kEpiQkv && a.S == 1) {
    fill_head_cache(a, rb, hcs, hpos, tid, kCW * 32);
    consumer_sync();
  }
  if (EPI == kEpiResid) {
    // consumer thread t owns output row t of the block (kCW * 32 == 128)
#pragma unroll
    for (int n = 0; n < NT * 8; ++n)
      if (n < a.batch) {
        const size_t o = (size_t)n * a.out_ld + (size_t)rb * kRowsPerBlock + tid;
        a.out[o] = __float2bfloat16_rn(__bfloat162float(rres[n]) + red[n * kRedLd + tid]);
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
      HeadPre hp;
      hp.p = hpos[task];
      hp.cs[0] = hcs[(task * 2) * 32 + lane];
      hp.cs[1] = hcs[(task * 2 + 1) * 32 + lane];
      if (a.d == 128)
        qkv_head_epilogue<4>(a, red, n, hl, hg, rn, hp);
      else
        qkv_head_epilogue<2>(a, red, n, hl, hg, rn, hp);
    }
  }
}

template <int NT, int EPI>
__global__ void __launch_bounds__(kThreads) proj_kernel(const ProjArgs a) {
  proj_body<NT, EPI>(a);
}

// Three or four batch tiles: at most 128 registers, so three CTAs share an SM.
template <int NT, int EPI>
__global__ void __maxnreg__(128) proj_kernel_wide(const ProjArgs a) {
  proj_body<NT, EPI>(a);
}

template <int NT, int EPI>
constexpr void (*proj_entry())(ProjArgs) {
  if constexpr (NT >= 3)
    return proj_kernel_wide<NT, EPI>;
  else
    return proj_kernel<NT, EPI>;
}

template <int NT, int EPI>
cudaError_t configure(int dev) {
  static unsigned long long configured = 0;  // one bit per device
  if (configured & (1ull << (dev & 63))) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(proj_entry<NT, EPI>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kProjMaxSmem);
  if (e != cudaSuccess) return e;
  // every kernel of the step asks for the maximum shared-memory carveout, so
  // CTAs of consecutive kernels can share an SM (programmatic overlap)
  e = cudaFuncSetAttribute(proj_entry<NT, EPI>(), cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  configured |= 1ull << (dev & 63);
  return cudaSuccess;
}

template <int NT, int EPI>
cudaError_t launch_one(const ProjArgs& a, int grid, size_t smem, cudaStream_t st, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure<NT, EPI>(dev);
  if (e != cudaSuccess) return e;
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
  return cudaLaunchKernelEx(&cfg, proj_entry<NT, EPI>(), a);
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

int resident_ctas(int nt, int epi, size_t smem) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  cudaError_t e = cudaSuccess;
#define FUTR_OCC(NT_, EPI_)                                                               \
  if (nt == NT_ && epi == EPI_) {                                                         \
    e = configure<NT_, EPI_>(dev);                                                        \
    if (e == cudaSuccess)                                                                 \
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, proj_entry<NT_, EPI_>(), kThreads, smem); \
  }
  FUTR_OCC(1, 0) FUTR_OCC(2, 0) FUTR_OCC(3, 0) FUTR_OCC(4, 0)
  FUTR_OCC(1, 1) FUTR_OCC(2, 1) FUTR_OCC(3, 1) FUTR_OCC(4, 1)
  FUTR_OCC(1, 2) FUTR_OCC(2, 2) FUTR_OCC(3, 2) FUTR_OCC(4, 2)
#undef FUTR_OCC
  return e == cudaSuccess ? n : 0;
}

}  // namespace

ProjPlan plan_projection(int rows, int cols, int batch, int n_sm, int force_split, int epi) {
  ProjPlan p{};
  p.n_rb = rows / kRowsPerBlock;
  p.n_groups = cols / kGroup;
  p.nt = (batch + 7) / 8;
  p.epi = epi;
  // ring stage = weight unit + activation tile; as deep as lets the target
  // number of CTAs share an SM (5 up to batch 8, else 3)
  p.stage_bytes = kUnitBytes + batch * kTileLd * 2;
  const int misc = 32 * 4 + 16 + 2 * kMaxRing * 8;
  const int per_sm = batch <= 8 ? 5 : 3;
  const int budget = 232448 / per_sm - 1024 - misc - 2048;  // per-CTA reserve and static arrays
  int ring = budget / p.stage_bytes;
  if (ring > kMaxRing) ring = kMaxRing;
  if (ring < 2) ring = 2;
  p.ring = ring;
  int ring_bytes = ring * p.stage_bytes;
  // the epilogue tile, the split-sum groups of small batches and (QKV) the
  // head tasks' RoPE factors alias the ring (up to 2 heads per row block)
  const int red_bytes = p.nt * 8 * kRedLd * 4 + kCW * 32 * 16 + (epi == kEpiQkv ? batch * 2 * 512 + 256 : 0);
  if (ring_bytes < red_bytes) ring_bytes = red_bytes;
  p.off_misc = (ring_bytes + 127) & ~127;
  p.smem = (size_t)p.off_misc + misc;
  // splits: balance waves of resident CTAs; each extra split costs a partial
  // write and a share of the reduction
  const int fit = resident_ctas(p.nt, epi, p.smem);
  const long long slots = (long long)n_sm * (fit > 0 ? fit : 1);
  int best_s = 1;
  double best = 1e30;
  for (int s = 1; s <= p.n_groups; ++s) {
    const long long items = (long long)p.n_rb * s;
    const long long waves = (items + slots - 1) / slots;
    const int per = (p.n_groups + s - 1) / s;
    const double cost = (double)waves * (per + 3) * (s > 1 ? 1.1 : 1.0);
    if (cost < best - 1e-9) {
      best = cost;
      best_s = s;
    }
  }
  if (force_split > 0) best_s = force_split < p.n_groups ? force_split : p.n_groups;
  p.S = best_s;
  p.rec_floats = batch * kRecLd;
  p.part_floats = (size_t)p.n_rb * p.S * p.rec_floats;
  return p;
}

cudaError_t launch_projection(int epi, const ProjPlan& p, ProjArgs a, cudaStream_t st, bool pdl) {
  a.S = p.S;
  a.n_groups = p.n_groups;
  a.ring = p.ring;
  a.stage_bytes = p.stage_bytes;
  a.off_misc = p.off_misc;
  a.rec_floats = p.rec_floats;
  const int grid = p.n_rb * p.S;
  if (epi == kEpiResid) return launch_nt<kEpiResid>(p.nt, a, grid, p.smem, st, pdl);
  if (epi == kEpiSwiglu) return launch_nt<kEpiSwiglu>(p.nt, a, grid, p.smem, st, pdl);
  return launch_nt<kEpiQkv>(p.nt, a, grid, p.smem, st, pdl);
}

}  // namespace futr
