// Persistent whole-block decode kernel: the five stages of one decode step
// (QKV with its fused epilogue, attention, O + residual, gate/up + SwiGLU,
// down + residual) in ONE launch.
//
// "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
// Hopper", abstract: decode time is spent reading the INT4 weights and the
// INT4 KV cache, with little reuse.  A launch per stage pays, five times per
// block, a launch, a pipeline fill and a split-K tail during which the weight
// stream stops.  Here the stream never stops: weights do not depend on the
// activations, so each CTA's weight producer streams the weight units of all
// its work items, stage after stage, into its shared-memory ring without ever
// waiting on another CTA; only the activation tiles (and the KV tiles of
// attention) wait for the previous stage to complete.
//
// Grid: C resident CTAs per SM, all resident at once: the kernel is launched
// in plain stream order (not programmatic), after the previous kernel has
// finished, and every cross-CTA wait is bounded.  A CTA has
//   warps 0..3  consumers: the products of each weight unit (unit_mma, the
//               same code as the one-projection kernels), the attention of
//               each KV tile (AttnWarp), the split-K / split-context tails and
//               the fused epilogues;
//   warp 4      lane 0, the weight producer: one 1-D bulk copy per weight
//               unit; for a KV tile only an L2 prefetch (the tile may still be
//               written); lane 1, the activation producer: per weight unit its
//               activation tile (2-D tensor copy), per KV tile its four bulk
//               copies, each phase only once the previous phase has completed
//               (the two lanes poll their barriers without blocking).
// Attention works in sub-groups of at most 4 query heads (one n-tile of hi|lo
// query columns), which keeps the consumers within the register budget of
// four CTAs per SM.
// A ring stage holds one weight unit + its activation tile, or one 64-position
// KV tile; its full barrier expects one arrival from each producer.
//
// Work: each projection phase's units (128 rows x 128 inputs) are split into
// equal contiguous ranges, one per CTA; a CTA's range covers parts of one or
// more row blocks.  Each part leaves a partial record; the last CTA to arrive
// at a row block adds the records (fixed order) and runs the epilogue, then
// counts the row block done.  Attention items are (context = sequence x
// kv-head x head sub-group, context range); each leaves (m, l, O) and the last
// arrival of a context merges its ranges in order, rotates back and stores o.
// Phase completion counters (row blocks / contexts done) gate the next phase;
// the last CTA to leave resets them for the next launch.
#include <cuda.h>

#include <algorithm>

#include "attn_dev.cuh"
#include "futr_internal.cuh"
#include "proj.cuh"
#include "proj_dev.cuh"

namespace futr {

namespace {

constexpr int kBlkCW = 4;                        // consumer warps
constexpr int kWarpP = kBlkCW;                   // the producer warp (lanes 0 and 1)
constexpr int kBlkThreads = (kBlkCW + 1) * 32;
constexpr int kBlkMaxRing = 32;
constexpr int kBlkMaxNC = 32;                   // context ranges per context
constexpr int kPhQ = 0, kPhA = 1;  // phases: QKV, attention, O (2), gate/up (3), down (4)
static_assert(kBlkCW == kCW && kBlkCW == kAttnCW, "one consumer thread per output row / four 16-position sub-tiles");

// misc area (after the scratch): ss [32] floats, flag [4] ints, full and
// empty barriers [kBlkMaxRing] each
constexpr int kBlkMisc = 32 * 4 + 16 + 2 * kBlkMaxRing * 8;

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait (bounded, abort-aware) until *cnt reaches `target` (acquire).
__device__ __forceinline__ bool wait_count(const unsigned* cnt, unsigned target, unsigned long long deadline,
                                           const int* err) {
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_gpu(cnt) >= target) return true;
    if ((i & 7u) == 7u && (global_ns() > deadline || aborted(err))) return false;
    __nanosleep(64);
  }
}

// The units of a projection phase: n_rb row blocks of n_groups units; `ne`
// CTAs take part, CTA c the units [lo(c), lo(c + 1)).
struct PhaseSplit {
  int n_rb, n_groups, ne;
  __device__ __forceinline__ long long units() const { return (long long)n_rb * n_groups; }
  __device__ __forceinline__ int lo(int c) const { return (int)((long long)c * units() / ne); }
  // the CTA whose range holds unit u
  __device__ __forceinline__ int owner(int u) const {
    int c = (int)(((long long)u * ne) / units());
    while (c + 1 < ne && lo(c + 1) <= u) ++c;
    while (c > 0 && lo(c) > u) --c;
    return c;
  }
};

// Context ranges of the attention phase: item j = (context j / NC, range j % NC);
// context = (sequence, kv-head, head sub-group).
struct AttnItem {
  int b, kvh, sub, r, L, t0, t1;
};

__device__ __forceinline__ AttnItem attn_item(const BlockArgs& a, int j) {
  AttnItem it;
  const int ctx = j / a.NC;
  it.r = j - ctx * a.NC;
  const int per_b = a.at.Hkv * a.nsub;
  it.b = ctx / per_b;
  it.kvh = (ctx - it.b * per_b) / a.nsub;
  it.sub = ctx - it.b * per_b - it.kvh * a.nsub;
  const int p = a.at.pos[it.b];
  it.L = p >= 0 && p < a.at.kv.cap ? p + 1 : 0;
  const int T = (it.L + kTilePos - 1) / kTilePos;
  it.t0 = (int)((long long)it.r * T / a.NC);
  it.t1 = (int)((long long)(it.r + 1) * T / a.NC);
  return it;
}

// phases Q, O, G, D are projections 0..3; the phase counter a projection's
// epilogues count, and the one its activation tiles wait for
constexpr int phase_of(int pi) { return pi == 0 ? kPhQ : pi + 1; }

template <int PI>
__device__ __forceinline__ PhaseSplit phase_split(const BlockArgs& a) {
  return PhaseSplit{a.ph[PI].n_rb, a.ph[PI].n_groups, a.ph[PI].ne};
}

// ------------------------------------------------------------- producer --
// One thread feeds the ring.  It walks this CTA's stage sequence (the units of
// its range in each projection phase, the KV tiles of its attention items)
// with two cursors: the weight cursor issues each weight unit's bulk copy (for
// a KV tile stage only its arrival and an L2 prefetch: the new token may not
// be written yet) and never waits on another CTA; the activation cursor issues
// each stage's activation tile or KV-tile copies once the phase before has
// completed.  Both advance in one loop of non-blocking tests, so neither can
// hold the other up.
struct Cursor {
  int seg;                  // 0 QKV, 1 attention, 2 O, 3 gate/up, 4 down, 5 past the end
  int u, u1;                // projection: the units [u, u1) still to go
  int j, t, t1, L, b, kvh;  // attention: item j, its tiles [t, t1)
};

__device__ __forceinline__ int seg_proj(int seg) { return seg == 0 ? 0 : seg - 1; }

// Move to the first stage at or after segment k.seg (attention: from item k.j).
__device__ __forceinline__ void cursor_settle(const BlockArgs& a, Cursor& k) {
  const int c = blockIdx.x;
  while (k.seg < 5) {
    if (k.seg == 1) {
      for (; k.j < a.n_ctx * a.NC; k.j += gridDim.x) {
        const AttnItem it = attn_item(a, k.j);
        if (it.t1 > it.t0) {
          k.t = it.t0;
          k.t1 = it.t1;
          k.L = it.L;
          k.b = it.b;
          k.kvh = it.kvh;
          return;
        }
      }
    } else {
      const BlockPhase& P = a.ph[seg_proj(k.seg)];
      const PhaseSplit sp{P.n_rb, P.n_groups, P.ne};
      if (c < sp.ne && sp.lo(c) < sp.lo(c + 1)) {
        k.u = sp.lo(c);
        k.u1 = sp.lo(c + 1);
        return;
      }
    }
    ++k.seg;
    k.j = c;
  }
}

__device__ __forceinline__ void cursor_next(const BlockArgs& a, Cursor& k) {
  if (k.seg == 1) {
    if (++k.t < k.t1) return;
    k.j += gridDim.x;
  } else {
    if (++k.u < k.u1) return;
    ++k.seg;
    k.j = blockIdx.x;
  }
  cursor_settle(a, k);
}

// Stage `s` of the ring is free again (its previous use was released).
__device__ __forceinline__ bool stage_free(const BlockArgs& a, uint64_t* empty, int s) {
  return s < a.ring || mbar_test_wait(&empty[s % a.ring], (uint32_t)((s / a.ring) + 1) & 1u);
}

template <int D>
__device__ __forceinline__ void issue_weight(const BlockArgs& a, const Cursor& k, int s, uint8_t* stages,
                                             uint64_t* full) {
  const int slot = s % a.ring;
  if (k.seg == 1) {
    mbar_arrive(&full[slot]);
    const uint8_t* strm = a.at.kv.stream(k.b, k.kvh);
    const int c0 = k.t * kTilePos, n16 = (min(kTilePos, k.L - c0) + 15) & ~15;
    l2_prefetch(strm + (size_t)c0 * (D / 2), (uint32_t)n16 * (D / 2));
    l2_prefetch(strm + (size_t)a.at.kv.cap * (D / 2) + (size_t)c0 * (D / 2), (uint32_t)n16 * (D / 2));
    return;
  }
  mbar_arrive_expect_tx(&full[slot], kUnitBytes);
  bulk_g2s(stages + (size_t)slot * a.stage_bytes, a.ph[seg_proj(k.seg)].w + (size_t)k.u * kUnitBytes, kUnitBytes,
           &full[slot]);
}

template <int D>
__device__ __forceinline__ void issue_act(const BlockArgs& a, const Cursor& k, int s, uint8_t* stages,
                                          uint64_t* full, const CUtensorMap* const* maps) {
  using Lay = AttnLayout<D>;
  const int slot = s % a.ring;
  uint8_t* st = stages + (size_t)slot * a.stage_bytes;
  if (k.seg == 1) {
    const uint8_t* strm = a.at.kv.stream(k.b, k.kvh);
    const int cap = a.at.kv.cap;
    const int c0 = k.t * kTilePos, n16 = (min(kTilePos, k.L - c0) + 15) & ~15;  // c0 + n16 <= cap
    const uint32_t cb = (uint32_t)n16 * (D / 2), sb = (uint32_t)n16 * 2;
    mbar_arrive_expect_tx(&full[slot], 2 * cb + 2 * sb);
    bulk_g2s(st, strm + (size_t)c0 * (D / 2), cb, &full[slot]);
    bulk_g2s(st + Lay::kCodes, strm + (size_t)cap * (D / 2) + (size_t)c0 * (D / 2), cb, &full[slot]);
    bulk_g2s(st + 2 * Lay::kCodes, strm + (size_t)cap * D + 2 * (size_t)c0, sb, &full[slot]);
    bulk_g2s(st + 2 * Lay::kCodes + 2 * kTilePos, strm + (size_t)cap * D + 2 * (size_t)cap + 2 * (size_t)c0, sb,
             &full[slot]);
    return;
  }
  const int pi = seg_proj(k.seg);
  mbar_arrive_expect_tx(&full[slot], (uint32_t)a.at.batch * kTileLd * 2);
  tma_2d_box(st + kUnitBytes, maps[pi], kGroup * (k.u % a.ph[pi].n_groups), 0, &full[slot]);
}

// Has the phase before segment `seg` completed (non-blocking, relaxed: the
// caller orders its copies after a fence once it has)?  QKV waits for
// nothing, attention for every QKV row block, O for every attention context,
// gate/up for O, down for gate/up.
__device__ __forceinline__ bool seg_ready(const BlockArgs& a, int seg) {
  if (seg == 0) return true;
  const unsigned target = seg == 1 ? (unsigned)a.ph[0].n_rb
                                   : (seg == 2 ? (unsigned)a.n_ctx : (unsigned)a.ph[seg - 2].n_rb);
  return ld_relaxed_gpu(&a.done[seg - 1]) >= target;
}

template <int D>
__device__ __forceinline__ void producer(const BlockArgs& a, const CUtensorMap* const* maps, uint8_t* stages,
                                         uint64_t* full, uint64_t* empty, int* flag) {
  for (int m = 0; m < 4; ++m) prefetch_map(maps[m]);
  // test hook (failure path): CTA 0 issues nothing, so its consumers' bounded
  // waits run out
  const bool hold = a.pa[0].withhold && blockIdx.x == 0;
  Cursor w{0, 0, 0, (int)blockIdx.x, 0, 0, 0, 0, 0};
  Cursor x = w;
  cursor_settle(a, w);
  cursor_settle(a, x);
  int wi = 0, xi = 0;
  bool ok = !hold;
  // the first ring's weights go out before the previous kernel has finished
  for (; ok && w.seg < 5 && wi < a.ring; ++wi, cursor_next(a, w)) issue_weight<D>(a, w, wi, stages, full);
  pdl_wait();  // x comes from the previous kernel
  const unsigned long long deadline = global_ns() + kWaitNs;
  bool x_ready = x.seg == 0;
  uint32_t idle = 0, poll = 0;
  while (ok && (w.seg < 5 || x.seg < 5)) {
    bool moved = false;
    // weights first: every free stage gets its unit at once
    while (w.seg < 5 && stage_free(a, empty, wi)) {
      issue_weight<D>(a, w, wi, stages, full);
      ++wi;
      cursor_next(a, w);
      moved = true;
    }
    if (x.seg < 5 && stage_free(a, empty, xi)) {
      // the phase counter is polled (relaxed, every few passes) only while
      // the activation cursor waits; once it is reached, one acquire fence
      // orders the copies after what the other CTAs wrote
      if (!x_ready && (poll++ & 7u) == 0 && seg_ready(a, x.seg)) {
        fence_acquire_gpu();
        fence_proxy_async_global();
        x_ready = true;
      }
      if (x_ready) {
        issue_act<D>(a, x, xi, stages, full, maps);
        ++xi;
        const int seg = x.seg;
        cursor_next(a, x);
        if (x.seg != seg) x_ready = x.seg == 0;
        moved = true;
      }
    }
    if (!moved && (++idle & 31u) == 0 && (global_ns() > deadline || aborted(a.err))) ok = false;
  }
  if (!ok && !hold) record_timeout(a.err);
  reinterpret_cast<volatile int*>(flag)[2] = wi;  // stages each cursor arrived on
  reinterpret_cast<volatile int*>(flag)[4] = xi;
  __threadfence_block();
  reinterpret_cast<volatile int*>(flag)[3] = 1;
}

// ------------------------------------------------------------ consumers --
// Ring position of the consumers (stage counter) and their status.
struct ConsumerState {
  int i;
  bool ok;
};

__device__ __forceinline__ bool take_stage(const BlockArgs& a, uint64_t* full, int s, unsigned long long deadline) {
  return mbar_wait_until(&full[s % a.ring], (uint32_t)(s / a.ring) & 1u, deadline, a.err);
}

__device__ __forceinline__ void give_stage(const BlockArgs& a, uint64_t* empty, int s) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[s % a.ring]);
}

// One attention item: context range it of context ctx; leaves its (m, l, O)
// record and, as the context's last range, merges the context.
template <int D, int NTQ>
__device__ __forceinline__ void attn_work(const BlockArgs& a, const AttnItem& it, int ctx, uint8_t* stages,
                                       float* scratch, int* flag, uint64_t* full, uint64_t* empty,
                                       unsigned long long deadline, ConsumerState& cs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.gc;  // heads per sub-group (at most 4)
  uint2* qf = reinterpret_cast<uint2*>(scratch);                       // [D/16][NTQ][32]
  float* cm = reinterpret_cast<float*>(qf + (D / 16) * NTQ * 32);      // [warps][G]
  float* cl = cm + kBlkCW * G;                                         // [warps][G]
  float* co = cl + kBlkCW * G;                                         // [warps][G][D]
  float* mO = co + kBlkCW * G * D;                                     // [G][D]
  float* mm = mO + G * D;                                              // [G]
  float* ml = mm + G;                                                  // [G]
  float* wgt = ml + G;                                                 // [kBlkMaxNC][G]
  const int hq0 = it.kvh * a.at.G + it.sub * G, Gv = min(G, a.at.G - it.sub * G);
  AttnWarp<D, NTQ> aw;
  aw.init();
  bool ok = true;
  if (it.t1 > it.t0) {
    build_qfrag<D, NTQ>(a.at.qrot + ((size_t)it.b * a.at.Hq + hq0) * D, Gv, qf, tid, kBlkCW * 32);
    consumer_sync();
    for (int t = it.t0; t < it.t1; ++t, ++cs.i) {
      if (!take_stage(a, full, cs.i, deadline)) {
        ok = false;
        break;
      }
      aw.tile(stages + (size_t)(cs.i % a.ring) * a.stage_bytes, min(kTilePos, it.L - t * kTilePos), qf,
              a.at.qk_scale_log2);
      give_stage(a, empty, cs.i);
    }
  }
  // every consumer warp learns whether some wait ran out before the next barrier
  if (!ok) flag[1] = 1;
  consumer_sync();
  if (flag[1]) {
    cs.ok = false;
    return;
  }
  aw.finish(cm, cl, co, G, Gv);
  consumer_sync();
  merge_warps(cm, cl, co, mO, mm, ml, wgt, G, Gv, D, tid, kBlkCW * 32, []() { consumer_sync(); });
  consumer_sync();
  // this range's record: m [G], l [G], O [G][D]
  float* rec = a.apart + ((size_t)ctx * a.NC + it.r) * a.arec_floats;
  for (int e = tid; e < Gv * D; e += kBlkCW * 32) rec[2 * G + e] = mO[e];
  if (tid < Gv) {
    rec[tid] = mm[tid];
    rec[G + tid] = ml[tid];
  }
  consumer_sync();
  if (tid == 0) flag[0] = atom_add_acq_rel_gpu(&a.actx[ctx], 1u) == (unsigned)(a.NC - 1) ? 1 : 0;
  consumer_sync();
  if (!flag[0]) return;
  // the last range of the context merges all of them, in range order
  const float* recs = a.apart + (size_t)ctx * a.NC * a.arec_floats;
  if (tid < Gv) {
    float M = -INFINITY;
    for (int r = 0; r < a.NC; ++r) M = fmaxf(M, __ldcg(recs + (size_t)r * a.arec_floats + tid));
    float Lr = 0.f;
    for (int r = 0; r < a.NC; ++r) {
      const float mr = __ldcg(recs + (size_t)r * a.arec_floats + tid);
      const float wt = mr == -INFINITY ? 0.f : exp2f(mr - M);
      wgt[r * G + tid] = wt;
      Lr += __ldcg(recs + (size_t)r * a.arec_floats + G + tid) * wt;
    }
    cm[tid] = Lr;
  }
  consumer_sync();
  for (int e = tid; e < Gv * D; e += kBlkCW * 32) {
    const int h = e / D;
    float acc = 0.f;
    for (int r = 0; r < a.NC; ++r) acc += wgt[r * G + h] * __ldcg(recs + (size_t)r * a.arec_floats + 2 * G + e);
    mO[e] = acc;
  }
  consumer_sync();
  for (int h = warp; h < Gv; h += kBlkCW) {
    const float inv = cm[h] > 0.f ? __fdiv_rn(1.0f, cm[h]) : 0.f;
    float v[D / 32];
#pragma unroll
    for (int q = 0; q < D / 32; ++q) v[q] = mO[h * D + lane + 32 * q] * inv;
    warp_fwht<D / 32>(v, a.at.nh, a.at.had_c);
    __nv_bfloat16* out = a.at.out + ((size_t)it.b * a.at.Hq + (size_t)hq0 + h) * D;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) out[lane + 32 * q] = __float2bfloat16_rn(v[q]);
  }
  if (it.L == 0 && it.kvh == 0 && it.sub == 0 && tid == 0) set_err(a.at.err, FUTR_ERR_OUT_OF_RANGE);
  if (tid == 0) a.actx[ctx] = 0u;  // self-reset for the next launch
  fence_proxy_async_global();      // o is read by other CTAs' tensor copies
  consumer_sync();
  if (tid == 0) red_release_add(&a.done[kPhA], 1u);
}

// One projection item: this CTA's units [ua, ub) of row block rb of
// projection PI (contributor `slot` of S), then the split-K tail and, as the
// last contributor, the epilogue.
template <int NT, int EPI, int PI>
__device__ __forceinline__ void proj_work(const BlockArgs& a, int rb, int ua, int ub, int S, int slot,
                                          uint8_t* stages, float* scratch, float* ss, int* flag, uint64_t* full,
                                          uint64_t* empty, unsigned long long deadline, ConsumerState& cs) {
  const int tid = threadIdx.x, lane = tid & 31;
  int xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = 8 * nt + (lane & 7);
    xrow[nt] = (n < a.at.batch ? n : 0) * kTileLd + 8 * (lane >> 3);
  }
  const int sq_off = (tid >> 4) * kTileLd + 8 * (tid & 15);
  float acc[kMT][NT][4];
#pragma unroll
  for (int m = 0; m < kMT; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][nt][e] = 0.f;
  float ssq[NT];
#pragma unroll
  for (int p = 0; p < NT; ++p) ssq[p] = 0.f;
  bool ok = true;
  for (int u = ua; u < ub; ++u, ++cs.i) {
    if (!take_stage(a, full, cs.i, deadline)) {
      ok = false;
      break;
    }
    unit_mma<NT, EPI != kEpiResid>(stages + (size_t)(cs.i % a.ring) * a.stage_bytes, xrow, sq_off, a.at.batch, acc,
                                   ssq);
    give_stage(a, empty, cs.i);
  }
  if (EPI != kEpiResid) ssq_to_smem<NT>(ssq, ss, a.at.batch);
  proj_tail<NT, EPI>(
      a.pa[PI], scratch, rb, S, slot, ss, flag, ok, [&](float* red) { acc_to_red<NT>(acc, red); },
      [&]() {
        fence_proxy_async_global();  // the outputs are read by other CTAs' tensor copies
        consumer_sync();
        if (tid == 0) red_release_add(&a.done[phase_of(PI)], 1u);
      });
  consumer_sync();  // the scratch is free again
  if (flag[1]) cs.ok = false;
}

// The consumers' part of projection phase PI: this CTA's part of each row
// block its unit range touches.
template <int NT, int EPI, int PI>
__device__ __forceinline__ void c_proj(const BlockArgs& a, uint8_t* stages, float* scratch, float* ss, int* flag,
                                       uint64_t* full, uint64_t* empty, unsigned long long deadline,
                                       ConsumerState& cs) {
  const PhaseSplit sp = phase_split<PI>(a);
  const int c = blockIdx.x;
  if (!cs.ok || c >= sp.ne) return;
  const int u0 = sp.lo(c), u1 = sp.lo(c + 1), ng = sp.n_groups;
  for (int rb = u0 / ng; rb * ng < u1 && cs.ok; ++rb) {
    const int first = sp.owner(rb * ng), last = sp.owner((rb + 1) * ng - 1);
    proj_work<NT, EPI, PI>(a, rb, max(u0, rb * ng), min(u1, (rb + 1) * ng), last - first + 1, c - first, stages,
                           scratch, ss, flag, full, empty, deadline, cs);
  }
}

template <int NT, int D>
__device__ __forceinline__ void consumers(const BlockArgs& a, uint8_t* stages, float* scratch, float* ss, int* flag,
                                          uint64_t* full, uint64_t* empty) {
  pdl_wait();
  const unsigned long long deadline = global_ns() + kWaitNs;
  ConsumerState cs{0, true};
  c_proj<NT, kEpiQkv, 0>(a, stages, scratch, ss, flag, full, empty, deadline, cs);
  // attention: after every QKV row block (rotated queries, new cache entries)
  bool qready = false;
  for (int j = blockIdx.x; j < a.n_ctx * a.NC && cs.ok; j += gridDim.x) {
    if (!qready) {
      // one thread waits for every QKV row block; the barrier passes its
      // outcome (and, through its acquire, the queries) to the others
      if (threadIdx.x == 0 && !wait_count(&a.done[kPhQ], (unsigned)a.ph[0].n_rb, deadline, a.err)) flag[1] = 1;
      consumer_sync();
      if (flag[1]) {
        cs.ok = false;
        break;
      }
      qready = true;
    }
    attn_work<D, 1>(a, attn_item(a, j), j / a.NC, stages, scratch, flag, full, empty, deadline, cs);
  }
  c_proj<NT, kEpiResid, 1>(a, stages, scratch, ss, flag, full, empty, deadline, cs);
  c_proj<NT, kEpiSwiglu, 2>(a, stages, scratch, ss, flag, full, empty, deadline, cs);
  c_proj<NT, kEpiResid, 3>(a, stages, scratch, ss, flag, full, empty, deadline, cs);
  if (!cs.ok) {
    record_timeout(a.err);
    flag[1] = 1;
  }
}

// Resident CTAs per SM the register budget is set for: three with one batch
// tile (at most 136 registers a thread), two with two.
template <int NT>
constexpr int kBlkPerSm = NT == 1 ? 3 : 2;

template <int NT, int D>
__global__ void __launch_bounds__(kBlkThreads, kBlkPerSm<NT>)
    block_kernel(const __grid_constant__ BlockArgs a, const __grid_constant__ CUtensorMap map_x,
                 const __grid_constant__ CUtensorMap map_o, const __grid_constant__ CUtensorMap map_h,
                 const __grid_constant__ CUtensorMap map_a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* stages = smem;
  float* scratch = reinterpret_cast<float*>(smem + a.off_scratch);
  float* ss = reinterpret_cast<float*>(smem + a.off_misc);  // [32] sums of squares per batch row
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.off_misc + 32 * 4 + 16);
  uint64_t* empty = full + kBlkMaxRing;
  // flags: [0] last arrival, [1] a consumer wait ran out; [2], [3] the weight
  // producer's stage count and stop; [4], [5] the activation producer's
  __shared__ int pflag[8];
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int k = 0; k < 8; ++k) pflag[k] = 0;
    for (int k = 0; k < a.ring; ++k) {
      mbar_init(&full[k], 2);  // one arrival from each producer
      mbar_init(&empty[k], kBlkCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kWarpP) {
    if ((tid & 31) == 0) {
      const CUtensorMap* maps[4] = {&map_x, &map_o, &map_h, &map_a};
      producer<D>(a, maps, stages, full, empty, pflag);
    }
  } else {
    consumers<NT, D>(a, stages, scratch, ss, pflag, full, empty);
  }
  __syncthreads();
  if (tid == 0) {
    if (pflag[1] || aborted(a.err)) {
      // a wait ran out somewhere: let this CTA's copies land before it exits.
      // A stage that one producer arrived on and the other did not never
      // completes: the missing arrival is made here.
      const int w = pflag[2], x = pflag[4];
      const int hi = max(w, x), lo = min(w, x);
      for (int s = max(lo, hi - a.ring); s < hi; ++s) mbar_arrive(&full[s % a.ring]);
      drain_ring(full, a.ring, hi);
    }
    // the last CTA to leave resets the phase counters for the next launch
    __threadfence();
    if (atom_add_acq_rel_gpu(&a.done[5], 1u) == gridDim.x - 1) {
      for (int k = 0; k < 6; ++k) a.done[k] = 0u;
      __threadfence();
    }
  }
}

template <int NT, int D>
cudaError_t configure_block(int dev) {
  static DeviceOnce configured;
  if (configured.done(dev)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(block_kernel<NT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kBlockMaxSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(block_kernel<NT, D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  configured.mark(dev);
  return cudaSuccess;
}

template <int NT, int D>
cudaError_t launch_t(const BlockPlan& p, const BlockArgs& a, const CUtensorMap* maps, cudaStream_t st, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure_block<NT, D>(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(kBlkThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  // Plain stream order, never programmatic launch: the CTAs of this grid wait
  // on one another, so all of them must be resident together, which a grid
  // launched early (its CTAs placed as the previous kernel's leave) does not
  // guarantee.  It also triggers no early launch of its successor.
  (void)pdl;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, block_kernel<NT, D>, a, maps[0], maps[1], maps[2], maps[3]);
}

template <int NT, int D>
int occupancy_t(size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (configure_block<NT, D>(dev) != cudaSuccess) {
    cudaGetLastError();  // not left pending for a later call to report
    return 0;
  }
  return remembered(occ_key(dev, 16 * NT + 1, D, smem), [&]() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, block_kernel<NT, D>, kBlkThreads, smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  });
}

// The instantiations: batch tiles 1..2 (batch <= 16), head dim 64 or 128.
#define FUTR_BLOCK_DISPATCH(NT_, D_, CALL)                   \
  do {                                                     \
    if (D_ == 128) {                                       \
      if (NT_ == 1) return CALL(1, 128);                   \
      return CALL(2, 128);                                 \
    }                                                      \
    if (NT_ == 1) return CALL(1, 64);                      \
    return CALL(2, 64);                                    \
  } while (0)

int occupancy_any(int nt, int D, size_t smem) {
#define FUTR_OCC_CALL(A, B) occupancy_t<A, B>(smem)
  FUTR_BLOCK_DISPATCH(nt, D, FUTR_OCC_CALL);
#undef FUTR_OCC_CALL
}

}  // namespace

BlockPlan plan_block(const futr_shape& s, int batch, int cap, int n_sm, int fixed_ctas_per_sm) {
  BlockPlan p{};
  if (batch < 1 || batch > kBlockMaxBatch) return p;
  // attention sub-groups of at most 4 query heads (one query n-tile)
  const int D = s.head_dim, G = s.n_q_heads / s.n_kv_heads, nsub = (G + 3) / 4, gc = (G + nsub - 1) / nsub,
            ntq = 1;
  p.nt = (batch + 7) / 8;
  p.ntq = ntq;
  p.nsub = nsub;
  p.gc = gc;
  // scratch: the projection epilogue (tile, split-sum groups, QKV RoPE factors)
  // or the attention work (query fragments, warp partials, merge), whichever
  // is larger
  const size_t proj_scr = (size_t)p.nt * 8 * kRedLd * 4 + kCW * 32 * 16 + (size_t)batch * 2 * 512 + 256;
  const size_t attn_scr = (size_t)(D / 16) * ntq * 32 * 8 +
                          4 * ((size_t)2 * kBlkCW * gc + (size_t)kBlkCW * gc * D + (size_t)gc * D + 2 * gc +
                               (size_t)kBlkMaxNC * gc);
  const size_t scratch = (std::max(proj_scr, attn_scr) + 127) & ~size_t(127);
  p.stage_bytes = (int)(std::max<size_t>(kUnitBytes + (size_t)batch * kTileLd * 2,
                                         D == 128 ? AttnLayout<128>::kStage : AttnLayout<64>::kStage) +
                        127) & ~127;
  // CTAs per SM: three up to batch 8, two beyond (or as asked); the ring as
  // deep as the shared memory left
  const int per_sm = fixed_ctas_per_sm > 0 ? fixed_ctas_per_sm : (batch <= 8 ? 3 : 2);
  const long long budget = std::min<long long>(232448 / per_sm - 1024, kBlockMaxSmem - 1024) - 128 -
                           (long long)scratch - kBlkMisc - 256;
  int ring = (int)(budget / p.stage_bytes);
  ring = std::min(ring, kBlkMaxRing);
  if (ring < 2) return BlockPlan{};
  p.ring = ring;
  p.off_scratch = ring * p.stage_bytes;
  p.off_misc = p.off_scratch + (int)scratch;
  p.smem = (size_t)p.off_misc + kBlkMisc + 128;  // the base is rounded up to 128 bytes
  const int fit = occupancy_any(p.nt, D, p.smem);
  const int ctas = std::min(per_sm, fit);
  p.grid = n_sm * std::max(ctas, 0);
  p.grid_cap = n_sm * per_sm;
  // context ranges: about one item per CTA, at most the tiles of the cache
  p.n_ctx = batch * s.n_kv_heads * p.nsub;
  const int tiles = (cap + kTilePos - 1) / kTilePos;
  p.NC = std::max(1, std::min({(std::max(p.grid, 1) + p.n_ctx - 1) / p.n_ctx, kBlkMaxNC, tiles}));
  p.arec_floats = 2 * gc + gc * D;
  p.ok = p.grid > 0;
  return p;
}

cudaError_t launch_block(const BlockPlan& p, const BlockArgs& a, const CUtensorMap* maps, cudaStream_t st, bool pdl) {
#define FUTR_LAUNCH_CALL(A, B) launch_t<A, B>(p, a, maps, st, pdl)
  FUTR_BLOCK_DISPATCH(p.nt, a.at.kv.d, FUTR_LAUNCH_CALL);
#undef FUTR_LAUNCH_CALL
}

}  // namespace futr
