// Device code of the W4A16 projections shared by the one-projection kernels
// (proj.cu) and the persistent whole-block kernel (block.cu): the consumer
// warps' products of one ring stage, the split-K tail (partial records,
// arrival, the last CTA's reduction) and the fused epilogues (residual,
// SwiGLU, QKV with RoPE, rotation and INT4 KV placement).
#pragma once

#include <cuda.h>

#include "futr_internal.cuh"
#include "proj.cuh"

namespace futr {
namespace {

constexpr int kCW = 4;                    // consumer warps
constexpr int kMT = 2;                    // 16-row MMA tiles per consumer warp
constexpr int kThreads = (kCW + 1) * 32;  // + producer warp
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

// One head task of the QKV epilogue for one warp: v holds the head's d sums
// times the RMSNorm factor (element lane + 32 j in v[j]); RoPE (q, k), the fp32
// rotation, then q' to qrot or k, v as INT4 + fp16 scale into cache slot p.
template <int J>
__device__ void qkv_head_core(const ProjArgs& a, float (&v)[J], int n, int hg, const HeadPre& pre) {
  constexpr int d = 32 * J;
  const int lane = threadIdx.x & 31;
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
  if (!FUTR_DCHECK(n < a.batch && hg < a.Hq + 2 * a.Hkv, a.err)) return;
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

// The same from the epilogue tile of the last CTA (global split-K tail).
template <int J>
__device__ void qkv_head_epilogue(const ProjArgs& a, const float* red, int n, int hl, int hg, float r,
                                  const HeadPre& pre) {
  constexpr int d = 32 * J;
  const int lane = threadIdx.x & 31;
  float v[J];
#pragma unroll
  for (int j = 0; j < J; ++j) v[j] = red[n * kRedLd + hl * d + lane + 32 * j] * r;
  qkv_head_core<J>(a, v, n, hg, pre);
}

// Position and RoPE factors of head hg for batch row n, as fill_head_cache
// stores them (q and k heads rotate by position; v heads get (1, 0)).
__device__ __forceinline__ HeadPre head_pre(const ProjArgs& a, int n, int hg) {
  const int lane = threadIdx.x & 31, half = a.d / 2;
  HeadPre hp;
  hp.p = a.pos[n];
  hp.cs[0] = hp.cs[1] = make_float2(1.f, 0.f);
  if (hg < a.Hq + a.Hkv) {
    const int pp = hp.p >= 0 && hp.p < a.kv.cap ? hp.p : 0;
    hp.cs[0] = a.rope[(size_t)pp * half + lane];
    if (half > 32) hp.cs[1] = a.rope[(size_t)pp * half + lane + 32];
  }
  return hp;
}

// The producer lane's count of issued ring stages, for the drain after a
// time-out: flag[2] = count, flag[3] = 1 once the producer has stopped.
__device__ __forceinline__ void publish_issued(int* flag, int issued) {
  reinterpret_cast<volatile int*>(flag)[2] = issued;
  __threadfence_block();
  reinterpret_cast<volatile int*>(flag)[3] = 1;
}

// After a time-out: wait (bounded) until the producer has stopped, then until
// the copies it issued into the ring have landed.  The ring's barriers and
// flags are found again from the shared-memory base (misc area at off_misc:
// 32 floats, 4 flag words, then the full barriers), so that nothing of the
// normal path stays live for this failure path.
__device__ __forceinline__ void drain_after_timeout(uint8_t* smem, int off_misc, int R) {
  volatile int* flag = reinterpret_cast<volatile int*>(smem + off_misc + 32 * 4);
  const unsigned long long dl = global_ns() + kWaitNs;
  while (flag[3] == 0 && global_ns() < dl) {
  }
  __threadfence_block();
  drain_ring(reinterpret_cast<uint64_t*>(smem + off_misc + 32 * 4 + 16), R, flag[2]);
}

__device__ __forceinline__ void tma_2d_box(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Pull a tensor map (a kernel parameter) into the copy engine's cache ahead of
// its first use.
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Activation tile of group g into a ring stage: one tensor copy of inputs
// 128 g .. 128 g + 135 of the batch rows, rows kTileLd elements apart (one
// row: its 128 inputs by a bulk copy).
template <bool kRow1>
__device__ __forceinline__ void issue_tile(const ProjArgs& a, const CUtensorMap* xmap, uint8_t* stage, int g,
                                           uint64_t* bar) {
  if (kRow1)
    bulk_g2s(stage + kUnitBytes, a.xin + (size_t)g * kGroup, kGroup * 2, bar);
  else
    tma_2d_box(stage + kUnitBytes, xmap, kGroup * g, 0, bar);
}

// Everything after the K-loop: the epilogue tile (filled by write_red from
// the caller's accumulators), the split record and arrival, the last CTA's
// reduction and the fused epilogue.  Consumer threads only.
// S CTAs contribute partial sums to row block rb (this one as contributor
// `slot`); their records sit at a.part + (rb * a.part_stride + s) * a.rec_floats.
// `red` is the epilogue scratch: the tile [NT*8][kRedLd], then the split-sum
// groups, then (QKV) the head tasks' RoPE factors.  done(): called by every
// consumer thread of the CTA that ran the epilogue, once its writes are issued.
// After a time-out (flag[1] set) it returns at once, writing nothing: the
// caller then lets its in-flight copies land (drain_after_timeout).
// pre (QKV, at most one head task per consumer warp): this warp's task's
// position and RoPE factors, loaded by the caller ahead of time; otherwise
// they are loaded during the arrival.
template <int NT, int EPI, class WriteRed, class Done>
__device__ __forceinline__ void proj_tail(const ProjArgs& a, float* red, int rb, int S, int slot, float* ss,
                                          int* flag, bool ok, WriteRed&& write_red, Done&& done,
                                          const HeadPre* pre = nullptr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the residual rows of this block (RESID): with one batch tile loaded now,
  // overlapping the split handshake; with more, in one burst after the
  // reduction, which keeps them out of its registers
  constexpr bool kEarly = NT == 1;
  __nv_bfloat16 rres[EPI == kEpiResid ? NT * 8 : 1];
  auto load_resid = [&]() {
    if (EPI == kEpiResid) {
#pragma unroll
      for (int n = 0; n < NT * 8; ++n)
        // through L2: in the whole-block kernel another CTA wrote it in this launch
        rres[n] = n < a.batch ? __ldcg(a.resid + (size_t)n * a.out_ld + (size_t)rb * kRowsPerBlock + tid)
                              : __float2bfloat16_rn(0.f);
    }
  };
  if (kEarly) load_resid();
  // QKV: the head tasks' positions and RoPE factors go to shared memory after
  // the epilogue tile and the split-sum groups (the ring is free by then)
  float2* hcs = reinterpret_cast<float2*>(red + NT * 8 * kRedLd + 4 * kCW * 32);
  int* hpos = reinterpret_cast<int*>(hcs + a.batch * (kRowsPerBlock / a.d) * 64);
  const bool have_pre = EPI == kEpiQkv && pre != nullptr && a.batch * (kRowsPerBlock / a.d) <= kCW;
  if (!ok) {
    record_timeout(a.err);
    flag[1] = 1;
  }
  // debug build: this CTA's split record and row block lie inside their regions
  if (tid == 0 && (S > 1 || EPI == kEpiQkvRec) &&
      !FUTR_DCHECK(rb < a.n_rb && slot < a.part_stride &&
                       ((size_t)rb * a.part_stride + a.part_stride) * a.rec_floats <= a.part_cap,
                   a.err))
    flag[1] = 1;

  // ------------------------------------------------------------ epilogue --
  consumer_sync();  // every warp is done with its accumulators (and, in a one-shot kernel, the ring)
  if (flag[1]) return;  // a wait ran out: write nothing (the arrival counters stay
                        // as they are: futr_check clears them with the time-out)
  write_red(red);
  consumer_sync();

  // records-only QKV: the record is all this kernel writes (the attention
  // kernel adds the records and runs the head epilogue)
  constexpr bool kDefer = EPI == kEpiQkvRec;
  if (S > 1 || kDefer) {
    // publish this split's partial record: per batch row 32 float4 of sums and
    // one float4 (sum of squares, 0, 0, 0); then count arrivals
    float* rec = a.part + ((size_t)rb * a.part_stride + slot) * a.rec_floats;
    const int items = a.batch * kRecCols;
    for (int e = tid; e < items; e += kCW * 32) {
      const int n = e / kRecCols, c4 = e - kRecCols * n;
      const float4 v = c4 < 32 ? reinterpret_cast<const float4*>(red + n * kRedLd)[c4]
                               : make_float4(EPI != kEpiResid ? ss[n] : 0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4*>(rec + n * kRecLd)[c4] = v;
    }
    if (kDefer) return;  // (the producer of CTA 0 checks the blob header)
    consumer_sync();
    if (tid == 0)
      flag[0] = atom_add_acq_rel_gpu(&a.cnt[rb], 1u) == (unsigned)(S - 1) ? 1 : 0;
    else if (EPI == kEpiQkv && !have_pre)
      fill_head_cache(a, rb, hcs, hpos, tid - 1, kCW * 32 - 1);  // overlaps the arrival
    consumer_sync();
    if (!flag[0]) return;
    // The last CTA adds the S records.  With few columns (small batch), G
    // groups of threads each add a contiguous range of splits, all loads of a
    // range in flight together; the G group sums are then added in group
    // order.  The order is fixed, so the result is deterministic.
    const int G = items >= kCW * 32 ? 1 : (kCW * 32) / items;
    float4* gsum = reinterpret_cast<float4*>(red + NT * 8 * kRedLd);  // [G][items], G > 1 only
    const float* part_rb = a.part + (size_t)rb * a.part_stride * a.rec_floats;
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
      for (int s0 = 0; s0 < S; s0 += kSP) {
        float4 v[kSP][kJ];
#pragma unroll
        for (int q = 0; q < kSP; ++q)
#pragma unroll
          for (int j = 0; j < kJ; ++j)
            if (col[j] >= 0 && s0 + q < S) v[q][j] = __ldcg(rec4 + (size_t)(s0 + q) * step + col[j]);
#pragma unroll
        for (int q = 0; q < kSP; ++q)
#pragma unroll
          for (int j = 0; j < kJ; ++j)
            if (col[j] >= 0 && s0 + q < S) {
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
      const int s_lo = grp * S / G, s_hi = (grp + 1) * S / G;
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
  if (EPI == kEpiQkv && S == 1 && !have_pre) {
    fill_head_cache(a, rb, hcs, hpos, tid, kCW * 32);
    consumer_sync();
  }
  if (EPI == kEpiResid) {
    // consumer thread t owns output row t of the block (kCW * 32 == 128)
#pragma unroll
    for (int n = 0; n < NT * 8; ++n)
      if (n < a.batch) {
        const size_t o = (size_t)n * a.out_ld + (size_t)rb * kRowsPerBlock + tid;
        if (FUTR_DCHECK(o < a.out_cap, a.err))
          a.out[o] = __float2bfloat16_rn(__bfloat162float(rres[n]) + red[n * kRedLd + tid]);
      }
  } else if (EPI == kEpiSwiglu) {
    for (int e = tid; e < a.batch * 64; e += kCW * 32) {
      const int n = e >> 6, r = e & 63;
      const float rn = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(ss[n], (float)a.K) + a.eps));
      const float g = rn * red[n * kRedLd + r];
      const float u = rn * red[n * kRedLd + 64 + r];
      const float sg = __fdiv_rn(g, 1.0f + expf(-g));
      const size_t o = (size_t)n * a.out_ld + (size_t)rb * 64 + r;
      if (FUTR_DCHECK(o < a.out_cap, a.err)) a.out[o] = __float2bfloat16_rn(sg * u);
    }
  } else if (EPI == kEpiQkv) {
    if (rb == 0 && tid == 0 && a.blob_magic && *a.blob_magic != kBlobMagic)
      set_err(a.err, FUTR_ERR_BAD_BLOB);
    const int hpr = kRowsPerBlock / a.d;
    for (int task = warp; task < a.batch * hpr; task += kCW) {
      const int n = task / hpr, hl = task % hpr;
      const int hg = rb * hpr + hl;
      const float rn = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(ss[n], (float)a.K) + a.eps));
      HeadPre hp;
      if (have_pre) {
        hp = *pre;  // task == warp
      } else {
        hp.p = hpos[task];
        hp.cs[0] = hcs[(task * 2) * 32 + lane];
        hp.cs[1] = hcs[(task * 2 + 1) * 32 + lane];
      }
      if (a.d == 128)
        qkv_head_epilogue<4>(a, red, n, hl, hg, rn, hp);
      else
        qkv_head_epilogue<2>(a, red, n, hl, hg, rn, hp);
    }
  }
  done();
}

// The products of one ring stage (a weight unit and its activation tile) for
// consumer warp `warp`'s 32 rows: per 16-row tile, acc += scale * (codes x
// tile), the codes unpacked in registers straight into bf16 MMA operands; with
// kSsq, also this thread's share of the tile's sum of squares (RMSNorm).
// xrow: ldmatrix row offsets of this lane's batch rows (elements); sq_off:
// this thread's 8 elements of the tile for the sum of squares.
template <int NT, bool kSsq>
__device__ __forceinline__ void unit_mma(const uint8_t* st, const int (&xrow)[NT], int sq_off, int batch,
                                         float (&acc)[kMT][NT][4], float (&ssq)[NT]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gr = lane >> 2;
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
  if (kSsq) {
#pragma unroll
    for (int p = 0; p < NT; ++p)
      if ((tid >> 4) + 8 * p < batch) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + sq_off + 8 * p * kTileLd);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(u[j] << 16), hi = __uint_as_float(u[j] & 0xffff0000u);
          ssq[p] = fmaf(lo, lo, fmaf(hi, hi, ssq[p]));
        }
      }
  }
}

// The accumulator fragments of consumer warp `warp` into the epilogue tile
// red[batch column][block row].
template <int NT>
__device__ __forceinline__ void acc_to_red(const float (&acc)[kMT][NT][4], float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gr = lane >> 2, t = lane & 3;
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

// The RMSNorm sums of squares of this thread's tile rows, reduced over the 16
// lanes of a half-warp (which cover a row), into ss[batch row].
template <int NT>
__device__ __forceinline__ void ssq_to_smem(float (&ssq)[NT], float* ss, int batch) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int p = 0; p < NT; ++p) {
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) ssq[p] += __shfl_xor_sync(0xffffffffu, ssq[p], o);
    const int n = (tid >> 4) + 8 * p;
    if ((tid & 15) == 0 && n < batch) ss[n] = ssq[p];
  }
}

}  // namespace
}  // namespace futr
