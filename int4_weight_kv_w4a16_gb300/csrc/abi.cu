// C ABI of libfutr.so (declared in include/futr.h): argument checking, memory
// layouts of the KV cache and the workspace, launch planning, and the five
// launches of one decode step.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include <nvtx3/nvToolsExt.h>

#include "futr_internal.cuh"
#include "proj.cuh"

using namespace futr;

namespace {

constexpr int kVersion = 10000;

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

// Per-stage NVTX ranges (FUTR_NVTX=1 in the environment, read once): a
// host-side range named for the stage around each kernel launch, for timeline
// tools.  Off by default.
bool nvtx_on();
struct Range {
  const bool on;
  explicit Range(const char* name) : on(nvtx_on()) {
    if (on) nvtxRangePushA(name);
  }
  ~Range() {
    if (on) nvtxRangePop();
  }
};

// Guard words: every region of a workspace and of a cache is followed by
// kGuardBytes of a fixed pattern (written at init, never by a kernel), so the
// guard of a region is the kGuardBytes just before the next region's start (the
// buffer's end for the last one).  futr_check compares them with the pattern:
// a kernel that wrote past the end of a region shows up as FUTR_ERR_CORRUPT.
constexpr uint64_t kGuardBytes = 256;
constexpr unsigned char kGuardByte = 0xA5;
constexpr uint32_t kGuardWord = 0xA5A5A5A5u;
constexpr int kMaxGuards = 16;
// the next region's start after one of `size` bytes at `off`
inline uint64_t after(uint64_t off, uint64_t size) { return align256(off + size) + kGuardBytes; }

bool shape_ok(const futr_shape* s) {
  if (!s) return false;
  const int d = s->head_dim;
  if (s->hidden <= 0 || s->hidden % 128) return false;
  if (d != 64 && d != 128) return false;
  if (s->n_q_heads <= 0 || s->n_kv_heads <= 0 || s->n_q_heads % s->n_kv_heads) return false;
  if (s->n_q_heads / s->n_kv_heads > 16) return false;
  if ((s->n_q_heads * d) % 128 || ((s->n_q_heads + 2 * s->n_kv_heads) * d) % 128) return false;
  if (s->inter <= 0 || s->inter % 128) return false;
  if (s->group != 128) return false;
  const int nh = s->had_block;
  if (nh < 2 || nh > d || (nh & (nh - 1))) return false;
  if (!(s->rms_eps > 0.f) || !(s->rope_theta > 0.f)) return false;
  return true;
}

bool same_shape(const futr_shape& a, const futr_shape& b) { return std::memcmp(&a, &b, sizeof(a)) == 0; }

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int env_int(const char* name) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : 0;
}

bool nvtx_on() {
  static const bool on = env_int("FUTR_NVTX") == 1;
  return on;
}

int round16(int c) { return (c + 15) & ~15; }

int env_int_or(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : dflt;
}

struct Plans {
  ProjPlan proj[4];  // QKV, O, GU, DOWN
  AttnPlan attn;
  BlockPlan blk;     // the persistent whole-block kernel (batch <= 16)
  // the five kernels: QKV writes its split records only (kEpiQkvRec) and the
  // attention kernel adds them and runs the head epilogue
  bool qkv_defer;
};

// Batches up to which the five kernels run the QKV head epilogue in the
// attention kernel.
constexpr int kQkvDeferMaxBatch = 32;

Plans plan_all(const futr_shape& s, int batch, int cap, int n_sm, int force, int force_attn, bool allow_defer) {
  const BlobSections sec = blob_sections(s);
  Plans p;
  const int epi[4] = {kEpiQkv, kEpiResid, kEpiSwiglu, kEpiResid};
  p.attn = plan_attention(s, batch, cap, n_sm, force_attn);
  // the QKV head epilogue in the attention kernel needs one cluster per
  // kv-head and sequence (so one CTA forms each new token)
  p.qkv_defer = allow_defer && batch <= kQkvDeferMaxBatch && p.attn.one_sub;
  for (int i = 0; i < 4; ++i)
    p.proj[i] = plan_projection(sec.rows[i], sec.cols[i], batch, n_sm, force,
                                i == 0 && p.qkv_defer ? kEpiQkvRec : epi[i]);
  p.blk = batch <= kBlockMaxBatch ? plan_block(s, batch, cap, n_sm, 0) : BlockPlan{};
  return p;
}

// Launch plans of one decode call.  FUTR_SPLITK / FUTR_ATTN_SPLIT force the
// split-K and context-range counts (within the planner's bounds);
// FUTR_QKV_DEFER=0 keeps the QKV head epilogue in the QKV kernel.
// Plans are kept per (shape, batch, capacity, SM count, these settings), so a
// repeated call only looks its plan up.
Plans make_plans(const futr_shape& s, int batch, int cap, int n_sm) {
  const int force = env_int("FUTR_SPLITK"), force_attn = env_int("FUTR_ATTN_SPLIT");
  const int defer = env_int_or("FUTR_QKV_DEFER", 1) != 0 ? 1 : 0;
  using Key = std::tuple<std::string, int, int, int, int, int, int>;
  static std::mutex mu;
  static std::map<Key, Plans> cache;
  const Key key(std::string(reinterpret_cast<const char*>(&s), sizeof(s)), batch, cap, n_sm, force, force_attn,
                defer);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const Plans p = plan_all(s, batch, cap, n_sm, force, force_attn, defer != 0);
  std::lock_guard<std::mutex> g(mu);
  if (cache.size() > 4096) cache.clear();
  return cache.emplace(key, p).first->second;
}

// Split records per row block that the persistent kernel's projection phase
// needs when `ne` CTAs share its n_rb x n_groups units in equal contiguous
// ranges: a row block of n_groups units meets at most n_groups / per + 2 of
// ranges of at least `per` units.
int block_stride(int n_rb, int n_groups, int ne) {
  const long long U = (long long)n_rb * n_groups;
  const int e = (int)std::min<long long>(ne, U);
  const int per = (int)(U / e);
  return std::min(e, n_groups / per + 2);
}

struct WsLayout {
  uint64_t err, qrot, o, h, a, xin, yout, pos, part, part_bytes, apart, apart_bytes, cnt, cnt_words, total;
};

WsLayout ws_layout(const futr_shape& s, int max_batch, int cap, int n_sm) {
  WsLayout L{};
  const uint64_t B = (uint64_t)max_batch;
  const uint64_t qd = (uint64_t)s.n_q_heads * s.head_dim;
  uint64_t off = 0;
  L.err = off; off = after(off, 16);
  L.qrot = off; off = after(off, B * qd * 4);
  L.o = off; off = after(off, B * qd * 2);
  L.h = off; off = after(off, B * s.hidden * 2);
  L.a = off; off = after(off, B * s.inter * 2);
  L.xin = off; off = after(off, B * s.hidden * 2);
  L.yout = off; off = after(off, B * s.hidden * 2);
  L.pos = off; off = after(off, B * 4);
  // split records: the largest any plan of a batch up to max_batch can use
  // (each projection's split cap, independent of occupancy answers and of
  // forced split counts)
  size_t part = 0, apart = 0;
  const BlobSections sec = blob_sections(s);
  uint64_t n_ctx_max = 0;
  for (int b = 1; b <= max_batch; ++b) {
    const Plans p = plan_all(s, b, cap, n_sm, 0, 0, true);
    for (int i = 0; i < 4; ++i)
      if ((p.proj[i].s_cap > 1 || p.proj[i].epi == kEpiQkvRec) && p.proj[i].part_cap_floats > part)
        part = p.proj[i].part_cap_floats;
    if (p.attn.part_floats > apart) apart = p.attn.part_floats;
    if (b <= kBlockMaxBatch) {
      // the persistent kernel with the most CTAs any plan of this batch uses
      const BlockPlan bp = plan_block(s, b, cap, n_sm, 0);
      if (bp.grid_cap > 0) {
        for (int i = 0; i < 4; ++i) {
          const int n_rb = sec.rows[i] / kRowsPerBlock, ng = sec.cols[i] / kGroup;
          const size_t f = (size_t)n_rb * block_stride(n_rb, ng, bp.grid_cap) * b * kRecLd;
          if (f > part) part = f;
        }
        const int tiles = (cap + 63) / 64;
        const int nc = std::max(1, std::min({(bp.grid_cap + bp.n_ctx - 1) / bp.n_ctx, 32, tiles}));
        const size_t af = (size_t)bp.n_ctx * nc * bp.arec_floats;
        if (af > apart) apart = af;
        if ((uint64_t)bp.n_ctx > n_ctx_max) n_ctx_max = bp.n_ctx;
      }
    }
  }
  L.part = off; L.part_bytes = part * 4; off = after(off, L.part_bytes);
  L.apart = off; L.apart_bytes = apart * 4; off = after(off, L.apart_bytes);
  // split-K arrival counters, one per row block of each projection; then the
  // persistent kernel's context counters and its six phase counters
  uint64_t cnt = 0;
  for (int i = 0; i < 4; ++i) cnt += sec.rows[i] / kRowsPerBlock;
  cnt += n_ctx_max + 6;
  L.cnt = off; L.cnt_words = cnt; off = after(off, cnt * 4);
  L.total = off;
  return L;
}

struct KvLayout {
  uint64_t stream_bytes, rope, err, total;
};

KvLayout kv_layout(const futr_shape& s, int n_layers, int max_batch, int cap16) {
  KvLayout L{};
  L.stream_bytes = kv_stream_bytes(cap16, s.head_dim);
  uint64_t off = after(0, (uint64_t)n_layers * max_batch * s.n_kv_heads * L.stream_bytes);
  L.rope = off;
  off = after(off, (uint64_t)cap16 * (s.head_dim / 2) * 8);
  L.err = off;
  L.total = after(off, 16);
  return L;
}

// Guard offsets of a workspace / cache described by `d` (see kGuardBytes).
int ws_guards(const futr_ws& d, uint64_t* g) {
  const uint64_t starts[] = {d.off_err, d.off_qrot, d.off_o, d.off_h, d.off_a, d.off_xin, d.off_yout,
                             d.off_pos, d.off_part, d.off_apart, d.off_cnt, d.bytes};
  int n = 0;
  for (size_t i = 1; i < sizeof(starts) / sizeof(starts[0]); ++i) g[n++] = starts[i] - kGuardBytes;
  return n;
}

int kv_guards(const futr_kv& d, uint64_t* g) {
  g[0] = d.rope_offset - kGuardBytes;
  g[1] = d.err_offset - kGuardBytes;
  g[2] = d.bytes - kGuardBytes;
  return 3;
}

cudaError_t fill_guards(void* base, const uint64_t* g, int n, cudaStream_t st) {
  for (int i = 0; i < n; ++i) {
    const cudaError_t e = cudaMemsetAsync(reinterpret_cast<uint8_t*>(base) + g[i], kGuardByte, kGuardBytes, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

struct GuardList {
  uint64_t off[kMaxGuards];
};

// One CTA per guard, one thread per word: a word off the pattern sets
// FUTR_ERR_CORRUPT in `err`.
__global__ void guard_check_kernel(const uint8_t* base, const GuardList g, int* err) {
  const uint32_t w = reinterpret_cast<const uint32_t*>(base + g.off[blockIdx.x])[threadIdx.x];
  if (w != kGuardWord) atomicCAS(err, 0, FUTR_ERR_CORRUPT);
}

cudaError_t check_guards(void* base, const uint64_t* g, int n, int* err, cudaStream_t st) {
  GuardList l{};
  for (int i = 0; i < n; ++i) l.off[i] = g[i];
  guard_check_kernel<<<n, (unsigned)(kGuardBytes / 4), 0, st>>>(reinterpret_cast<const uint8_t*>(base), l, err);
  return cudaGetLastError();
}

bool kv_ok(const futr_kv* kv) { return kv && kv->magic == kKvMagic && kv->base; }
bool ws_ok(const futr_ws* ws) { return ws && ws->magic == kWsMagic && ws->base; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

template <class T>
T* at(void* base, uint64_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(base) + off);
}

futr_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FUTR_OK : FUTR_ERR_CUDA; }

// Shared argument checks of the decode entry points.
futr_status check_decode(const void* blob, const futr_kv* kv, int layer, int batch, const futr_ws* ws) {
  if (!blob || !kv_ok(kv) || !ws_ok(ws)) return FUTR_ERR_INVALID_ARG;
  if (!same_shape(kv->shape, ws->shape)) return FUTR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= kv->n_layers) return FUTR_ERR_INVALID_ARG;
  if (batch < 1 || batch > kMaxBatch) return FUTR_ERR_UNSUPPORTED;
  if (batch > kv->max_batch || batch > ws->max_batch) return FUTR_ERR_INVALID_ARG;
  if (kv->capacity > ws->capacity) return FUTR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(blob) & 15) != 0) return FUTR_ERR_INVALID_ARG;
  return FUTR_OK;
}

// Use the persistent whole-block kernel for this call?  Only when asked for
// (FUTR_PERSISTENT=1): measured slower than the five kernels on the 8B and
// 70B blocks, it stays an option, not the default.
bool use_block_kernel(const Plans& P, int batch) {
  return batch <= kBlockMaxBatch && P.blk.ok && env_int_or("FUTR_PERSISTENT", 0) != 0;
}

// One decode step: the persistent whole-block kernel (batch <= 16), or five
// kernels with programmatic dependent launch.  events: NULL, or 6 events
// recorded around the five kernels (then launched without programmatic
// overlap, always as five kernels).
futr_status run_block(const uint16_t* x, const void* blob, const futr_kv* kv, int layer, int batch,
                      const int32_t* pos, uint16_t* y, const futr_ws* ws, cudaStream_t st,
                      cudaEvent_t* events) {
  const futr_shape& s = ws->shape;
  const Plans P = make_plans(s, batch, kv->capacity, ws->n_sm);
  const BlobSections sec = blob_sections(s);
  const uint8_t* wb = reinterpret_cast<const uint8_t*>(blob);
  void* base = ws->base;
  int* err = at<int>(base, ws->off_err);
  unsigned* cnt = at<unsigned>(base, ws->off_cnt);
  float* part = at<float>(base, ws->off_part);
  float* qrot = at<float>(base, ws->off_qrot);
  __nv_bfloat16* o = at<__nv_bfloat16>(base, ws->off_o);
  __nv_bfloat16* h = at<__nv_bfloat16>(base, ws->off_h);
  __nv_bfloat16* a = at<__nv_bfloat16>(base, ws->off_a);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(y);
  const bool pdl = events == nullptr;
  const KvView kvl = kv_layer_view(*kv, layer);
  const float had_c = (float)(1.0 / std::sqrt((double)s.had_block));

  // the four projections' arguments: QKV (S2), O (S4), gate/up (S5), down (S6)
  ProjArgs PA[4];
  const __nv_bfloat16* xin[4] = {xb, o, h, a};
  const __nv_bfloat16* resid[4] = {nullptr, xb, nullptr, h};
  __nv_bfloat16* outs[4] = {nullptr, h, a, yb};
  const int out_ld[4] = {0, s.hidden, s.inter, s.hidden};
  unsigned* cnt_next = cnt;
  for (int i = 0; i < 4; ++i) {
    ProjArgs A{};
    A.w = wb + sec.off[i];
    A.xin = xin[i];
    A.K = sec.cols[i];
    A.batch = batch;
    A.part = part;
    A.err = err;
    A.eps = s.rms_eps;
    A.cnt = cnt_next;
    cnt_next += sec.rows[i] / kRowsPerBlock;
    A.resid = resid[i];
    A.out = outs[i];
    A.out_ld = out_ld[i];
    A.n_rb = sec.rows[i] / kRowsPerBlock;
    A.part_cap = ws->part_bytes / 4;
    A.out_cap = (size_t)batch * out_ld[i];
#ifdef FUTR_DEBUG
    // FUTR_TEST_SHRINK_OUT=1 (debug build, tests of the bounds checks only):
    // the outputs of O, gate/up and down are checked against a region of one
    // element, so their first writes fail the check and are skipped
    if (env_int("FUTR_TEST_SHRINK_OUT") == 1 && i > 0) A.out_cap = 1;
#endif
    if (i == 0) {
      A.blob_magic = reinterpret_cast<const uint64_t*>(blob);
      A.qrot = qrot;
      A.kv = kvl;
      A.pos = pos;
      A.rope = at<const float2>(kv->base, kv->rope_offset);
      A.Hq = s.n_q_heads;
      A.Hkv = s.n_kv_heads;
      A.d = s.head_dim;
      A.nh = s.had_block;
      A.had_c = had_c;
      // FUTR_TEST_WITHHOLD_COPY=1 (tests of the failure path only): the first
      // CTA of the QKV projection issues no copy, so its bounded waits run
      // out and the step reports FUTR_ERR_TIMEOUT
      A.withhold = env_int("FUTR_TEST_WITHHOLD_COPY") == 1 ? 1 : 0;
    }
    PA[i] = A;
  }
  AttnArgs AT{};
  AT.qrot = qrot;
  AT.kv = kvl;
  AT.pos = pos;
  AT.batch = batch;
  AT.Hq = s.n_q_heads;
  AT.Hkv = s.n_kv_heads;
  AT.G = s.n_q_heads / s.n_kv_heads;
  AT.nh = s.had_block;
  AT.qk_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.head_dim));
  AT.had_c = had_c;
  AT.out = o;
  AT.err = err;

  if (!events && use_block_kernel(P, batch)) {
    const BlockPlan& bp = P.blk;
    BlockArgs B{};
    for (int i = 0; i < 4; ++i) {
      const int n_rb = sec.rows[i] / kRowsPerBlock, ng = sec.cols[i] / kGroup;
      const long long U = (long long)n_rb * ng;
      B.pa[i] = PA[i];
      B.pa[i].rec_floats = batch * kRecLd;
      B.ph[i].w = PA[i].w;
      B.ph[i].n_rb = n_rb;
      B.ph[i].n_groups = ng;
      B.ph[i].ne = (int)std::min<long long>(bp.grid, U);
      B.pa[i].part_stride = block_stride(n_rb, ng, B.ph[i].ne);
      if ((size_t)n_rb * B.pa[i].part_stride * B.pa[i].rec_floats * 4 > ws->part_bytes) return FUTR_ERR_INVALID_ARG;
    }
    B.at = AT;
    B.n_ctx = bp.n_ctx;
    B.NC = bp.NC;
    B.nsub = bp.nsub;
    B.gc = bp.gc;
    B.arec_floats = bp.arec_floats;
    if ((size_t)bp.n_ctx * bp.NC * bp.arec_floats * 4 > ws->apart_bytes) return FUTR_ERR_INVALID_ARG;
    B.apart = at<float>(base, ws->off_apart);
    B.actx = cnt_next;
    B.done = cnt_next + (size_t)batch * s.n_kv_heads * bp.nsub;
    if ((uint64_t)(B.done + 6 - cnt) > ws->cnt_words) return FUTR_ERR_INVALID_ARG;
    B.ring = bp.ring;
    B.stage_bytes = bp.stage_bytes;
    B.off_scratch = bp.off_scratch;
    B.off_misc = bp.off_misc;
    B.err = err;
    CUtensorMap maps[4];
    for (int i = 0; i < 4; ++i)
      if (!make_proj_tile_map(&maps[i], xin[i], batch, sec.cols[i], batch)) return FUTR_ERR_CUDA;
    Range r("futr.block");
    return cuda_status(launch_block(bp, B, maps, st, pdl));
  }

  for (int i = 0; i < 4; ++i)
    if ((P.proj[i].S > 1 || P.proj[i].epi == kEpiQkvRec) && P.proj[i].part_floats * 4 > ws->part_bytes)
      return FUTR_ERR_INVALID_ARG;
  if (P.attn.part_floats * 4 > ws->apart_bytes) return FUTR_ERR_INVALID_ARG;
  if (P.qkv_defer) {
    // QKV leaves its records (in `part`, which O overwrites only after the
    // attention kernel has completed) to the attention kernel
    AT.qkv_part = part;
    AT.qkv_S = P.proj[0].S;
    AT.qkv_stride = P.proj[0].S;
    AT.qkv_rec_floats = P.proj[0].rec_floats;
    AT.qkv_part_cap = ws->part_bytes / 4;
    AT.hidden = s.hidden;
    AT.eps = s.rms_eps;
    AT.rope = PA[0].rope;
  }
  static const char* const names[4] = {"futr.qkv", "futr.o", "futr.gate_up", "futr.down"};
  cudaError_t e;
  for (int i = 0; i < 4; ++i) {
    if (events) cudaEventRecord(events[i == 0 ? 0 : i + 1], st);
    {
      Range r(names[i]);
      e = launch_projection(P.proj[i].epi, P.proj[i], PA[i], st, pdl);
    }
    if (e != cudaSuccess) return FUTR_ERR_CUDA;
    if (i == 0) {
      // S3: attention
      if (events) cudaEventRecord(events[1], st);
      Range r("futr.attention");
      e = launch_attention(P.attn, AT, s.head_dim, st, pdl);
      if (e != cudaSuccess) return FUTR_ERR_CUDA;
    }
  }
  if (events) cudaEventRecord(events[5], st);
  return FUTR_OK;
}

// The device address of page-locked host memory that the device can access
// (mapped), or nullptr for any other pointer.
void* mapped_ptr(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

}  // namespace

extern "C" {

const char* futr_status_string(futr_status s) {
  switch (s) {
    case FUTR_OK: return "ok";
    case FUTR_ERR_INVALID_ARG: return "invalid argument";
    case FUTR_ERR_UNSUPPORTED: return "unsupported shape or batch";
    case FUTR_ERR_CUDA: return "CUDA error";
    case FUTR_ERR_OUT_OF_RANGE: return "position outside the KV cache";
    case FUTR_ERR_TIMEOUT: return "device wait timed out";
    case FUTR_ERR_BAD_BLOB: return "weight blob header mismatch";
    case FUTR_ERR_NOT_PD: return "dampened Hessian not positive definite";
    case FUTR_ERR_CORRUPT: return "guard words after a workspace or cache region overwritten";
    case FUTR_ERR_BOUNDS: return "device bounds check failed (debug build)";
    default: return "unknown status";
  }
}

int32_t futr_version(void) { return kVersion; }

futr_status futr_weights_size(const futr_shape* shape, size_t* bytes) {
  if (!bytes) return FUTR_ERR_INVALID_ARG;
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  *bytes = (size_t)blob_sections(*shape).total;
  return FUTR_OK;
}

futr_status futr_pack_weights(const futr_shape* shape, const float* wq, const float* wk, const float* wv,
                              const float* wo, const float* wgate, const float* wup, const float* wdown,
                              const float* g_attn, const float* g_mlp, void* blob, size_t blob_bytes,
                              void* stream) {
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  if (!wq || !wk || !wv || !wo || !wgate || !wup || !wdown || !g_attn || !g_mlp || !blob)
    return FUTR_ERR_INVALID_ARG;
  if (blob_bytes < blob_sections(*shape).total || (reinterpret_cast<uintptr_t>(blob) & 255))
    return FUTR_ERR_INVALID_ARG;
  return cuda_status(launch_pack(*shape, wq, wk, wv, wo, wgate, wup, wdown, g_attn, g_mlp,
                                 reinterpret_cast<uint8_t*>(blob), as_stream(stream)));
}

futr_status futr_gptq_scratch_size(const futr_shape* shape, size_t* bytes) {
  if (!bytes) return FUTR_ERR_INVALID_ARG;
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  *bytes = gptq_scratch_bytes(*shape);
  return FUTR_OK;
}

futr_status futr_pack_weights_gptq(const futr_shape* shape, const float* wq, const float* wk, const float* wv,
                                   const float* wo, const float* wgate, const float* wup, const float* wdown,
                                   const float* g_attn, const float* g_mlp, const double* h_attn,
                                   const double* h_o, const double* h_mlp, const double* h_down, double damp,
                                   void* scratch, size_t scratch_bytes, void* blob, size_t blob_bytes,
                                   void* stream) {
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  if (!wq || !wk || !wv || !wo || !wgate || !wup || !wdown || !g_attn || !g_mlp || !blob || !h_attn || !h_o ||
      !h_mlp || !h_down || !scratch)
    return FUTR_ERR_INVALID_ARG;
  if (!(damp > 0.0) || !std::isfinite(damp)) return FUTR_ERR_INVALID_ARG;
  if (blob_bytes < blob_sections(*shape).total || (reinterpret_cast<uintptr_t>(blob) & 255))
    return FUTR_ERR_INVALID_ARG;
  if (scratch_bytes < gptq_scratch_bytes(*shape) || (reinterpret_cast<uintptr_t>(scratch) & 255))
    return FUTR_ERR_INVALID_ARG;
  int bad = 0;
  const futr_status st = cuda_status(launch_pack_gptq(*shape, wq, wk, wv, wo, wgate, wup, wdown, g_attn, g_mlp,
                                                      h_attn, h_o, h_mlp, h_down, damp, scratch,
                                                      reinterpret_cast<uint8_t*>(blob), &bad, as_stream(stream)));
  if (st != FUTR_OK) return st;
  return bad ? FUTR_ERR_NOT_PD : FUTR_OK;
}

futr_status futr_unpack_weights(const futr_shape* shape, const void* blob, int32_t which, int8_t* codes,
                                uint16_t* scales, void* stream) {
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  if (!blob || !codes || !scales || which < FUTR_PROJ_QKV || which > FUTR_PROJ_DOWN) return FUTR_ERR_INVALID_ARG;
  return cuda_status(launch_unpack(*shape, reinterpret_cast<const uint8_t*>(blob), which, codes, scales,
                                   as_stream(stream)));
}

futr_status futr_kv_size(const futr_shape* shape, int32_t n_layers, int32_t max_batch, int32_t capacity,
                         size_t* bytes) {
  if (!bytes) return FUTR_ERR_INVALID_ARG;
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  if (n_layers < 1 || max_batch < 1 || capacity < 1) return FUTR_ERR_INVALID_ARG;
  if (capacity > kMaxCapacity) return FUTR_ERR_UNSUPPORTED;
  *bytes = (size_t)kv_layout(*shape, n_layers, max_batch, round16(capacity)).total;
  return FUTR_OK;
}

futr_status futr_kv_init(const futr_shape* shape, int32_t n_layers, int32_t max_batch, int32_t capacity,
                         void* kv_mem, size_t kv_bytes, futr_kv* kv, void* stream) {
  if (!kv || !kv_mem) return FUTR_ERR_INVALID_ARG;
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  if (n_layers < 1 || max_batch < 1 || capacity < 1) return FUTR_ERR_INVALID_ARG;
  if (capacity > kMaxCapacity) return FUTR_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(kv_mem) & 255) return FUTR_ERR_INVALID_ARG;
  const int cap = round16(capacity);
  const KvLayout L = kv_layout(*shape, n_layers, max_batch, cap);
  if (kv_bytes < L.total) return FUTR_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaMemsetAsync(kv_mem, 0, L.total, st);
  if (e != cudaSuccess) return FUTR_ERR_CUDA;
  e = launch_rope_table(at<float2>(kv_mem, L.rope), cap, shape->head_dim, shape->rope_theta, st);
  if (e != cudaSuccess) return FUTR_ERR_CUDA;
  futr_kv d{};
  d.shape = *shape;
  d.n_layers = n_layers;
  d.max_batch = max_batch;
  d.capacity = cap;
  d.base = kv_mem;
  d.bytes = L.total;
  d.stream_bytes = L.stream_bytes;
  d.rope_offset = L.rope;
  d.err_offset = L.err;
  d.magic = kKvMagic;
  uint64_t g[kMaxGuards];
  if (fill_guards(kv_mem, g, kv_guards(d, g), st) != cudaSuccess) return FUTR_ERR_CUDA;
  *kv = d;
  return FUTR_OK;
}

futr_status futr_kv_append(const futr_kv* kv, int32_t layer, int32_t seq0, int32_t batch, const int32_t* pos,
                           int32_t n_tok, const uint16_t* k, const uint16_t* v, void* stream) {
  if (!kv_ok(kv) || !pos || !k || !v) return FUTR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= kv->n_layers || batch < 1 || seq0 < 0 || seq0 + batch > kv->max_batch)
    return FUTR_ERR_INVALID_ARG;
  if (n_tok < 1 || n_tok > kv->capacity) return FUTR_ERR_INVALID_ARG;
  return cuda_status(launch_kv_append(*kv, layer, seq0, batch, pos, n_tok, k, v,
                                      at<int>(kv->base, kv->err_offset), as_stream(stream)));
}

futr_status futr_kv_read(const futr_kv* kv, int32_t layer, int32_t seq, int32_t n_pos, int8_t* k_codes,
                         uint16_t* k_scales, int8_t* v_codes, uint16_t* v_scales, void* stream) {
  if (!kv_ok(kv) || !k_codes || !k_scales || !v_codes || !v_scales) return FUTR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= kv->n_layers || seq < 0 || seq >= kv->max_batch) return FUTR_ERR_INVALID_ARG;
  if (n_pos < 1 || n_pos > kv->capacity) return FUTR_ERR_INVALID_ARG;
  return cuda_status(launch_kv_read(*kv, layer, seq, n_pos, k_codes, k_scales, v_codes, v_scales,
                                    as_stream(stream)));
}

futr_status futr_workspace_size(const futr_shape* shape, int32_t max_batch, int32_t capacity, size_t* bytes) {
  if (!bytes) return FUTR_ERR_INVALID_ARG;
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  if (max_batch < 1 || max_batch > kMaxBatch || capacity < 1) return FUTR_ERR_INVALID_ARG;
  if (capacity > kMaxCapacity) return FUTR_ERR_UNSUPPORTED;
  const int n_sm = current_sm_count();
  if (n_sm <= 0) return FUTR_ERR_CUDA;
  *bytes = (size_t)ws_layout(*shape, max_batch, round16(capacity), n_sm).total;
  return FUTR_OK;
}

futr_status futr_workspace_init(const futr_shape* shape, int32_t max_batch, int32_t capacity, void* ws_mem,
                                size_t ws_bytes, futr_ws* ws, void* stream) {
  if (!ws || !ws_mem) return FUTR_ERR_INVALID_ARG;
  if (!shape_ok(shape)) return FUTR_ERR_UNSUPPORTED;
  if (max_batch < 1 || max_batch > kMaxBatch || capacity < 1) return FUTR_ERR_INVALID_ARG;
  if (capacity > kMaxCapacity) return FUTR_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(ws_mem) & 255) return FUTR_ERR_INVALID_ARG;
  const int n_sm = current_sm_count();
  if (n_sm <= 0) return FUTR_ERR_CUDA;
  const int cap = round16(capacity);
  const WsLayout L = ws_layout(*shape, max_batch, cap, n_sm);
  if (ws_bytes < L.total) return FUTR_ERR_INVALID_ARG;
  if (cudaMemsetAsync(ws_mem, 0, L.total, as_stream(stream)) != cudaSuccess) return FUTR_ERR_CUDA;
  futr_ws d{};
  d.shape = *shape;
  d.max_batch = max_batch;
  d.capacity = cap;
  d.n_sm = n_sm;
  d.base = ws_mem;
  d.bytes = L.total;
  d.off_err = L.err;
  d.off_qrot = L.qrot;
  d.off_o = L.o;
  d.off_h = L.h;
  d.off_a = L.a;
  d.off_xin = L.xin;
  d.off_yout = L.yout;
  d.off_pos = L.pos;
  d.off_part = L.part;
  d.part_bytes = L.part_bytes;
  d.off_apart = L.apart;
  d.apart_bytes = L.apart_bytes;
  d.off_cnt = L.cnt;
  d.cnt_words = L.cnt_words;
  d.magic = kWsMagic;
  uint64_t g[kMaxGuards];
  if (fill_guards(ws_mem, g, ws_guards(d, g), as_stream(stream)) != cudaSuccess) return FUTR_ERR_CUDA;
  *ws = d;
  return FUTR_OK;
}

futr_status futr_decode_block(const uint16_t* x, const void* blob, const futr_kv* kv, int32_t layer,
                              int32_t batch, const int32_t* pos, uint16_t* y, const futr_ws* ws, void* stream) {
  if (!x || !pos || !y || x == y) return FUTR_ERR_INVALID_ARG;
  const futr_status st = check_decode(blob, kv, layer, batch, ws);
  if (st != FUTR_OK) return st;
  return run_block(x, blob, kv, layer, batch, pos, y, ws, as_stream(stream), nullptr);
}

futr_status futr_decode_block_timed(const uint16_t* x, const void* blob, const futr_kv* kv, int32_t layer,
                                    int32_t batch, const int32_t* pos, uint16_t* y, const futr_ws* ws,
                                    void* stream, float* stage_ms_host) {
  if (!x || !pos || !y || x == y || !stage_ms_host) return FUTR_ERR_INVALID_ARG;
  futr_status st = check_decode(blob, kv, layer, batch, ws);
  if (st != FUTR_OK) return st;
  cudaEvent_t ev[6];
  for (int i = 0; i < 6; ++i)
    if (cudaEventCreate(&ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      return FUTR_ERR_CUDA;
    }
  cudaStream_t s = as_stream(stream);
  st = run_block(x, blob, kv, layer, batch, pos, y, ws, s, ev);
  if (st == FUTR_OK && cudaStreamSynchronize(s) != cudaSuccess) st = FUTR_ERR_CUDA;
  for (int i = 0; i < 5 && st == FUTR_OK; ++i)
    if (cudaEventElapsedTime(&stage_ms_host[i], ev[i], ev[i + 1]) != cudaSuccess) st = FUTR_ERR_CUDA;
  for (int i = 0; i < 6; ++i) cudaEventDestroy(ev[i]);
  return st;
}

futr_status futr_decode_block_host(const uint16_t* x_host, const void* blob, const futr_kv* kv, int32_t layer,
                                   int32_t batch, const int32_t* pos_host, uint16_t* y_host, const futr_ws* ws,
                                   void* stream) {
  if (!x_host || !pos_host || !y_host) return FUTR_ERR_INVALID_ARG;
  futr_status st = check_decode(blob, kv, layer, batch, ws);
  if (st != FUTR_OK) return st;
  cudaStream_t s = as_stream(stream);
  const size_t xb = (size_t)batch * ws->shape.hidden * 2;
  uint16_t* xd = at<uint16_t>(ws->base, ws->off_xin);
  uint16_t* yd = at<uint16_t>(ws->base, ws->off_yout);
  int32_t* pd = at<int32_t>(ws->base, ws->off_pos);
  if (cudaMemcpyAsync(xd, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) return FUTR_ERR_CUDA;
  // pinned (page-locked, device-mapped) pos and y: the kernels read pos and
  // write y in host memory directly (plain loads and stores), which saves two
  // copies per call; otherwise both go through the workspace's staging rows
  const int32_t* pos_dev = static_cast<const int32_t*>(mapped_ptr(pos_host));
  uint16_t* y_dev = static_cast<uint16_t*>(mapped_ptr(y_host));
  const bool direct = pos_dev && y_dev;
  if (!direct && cudaMemcpyAsync(pd, pos_host, (size_t)batch * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FUTR_ERR_CUDA;
  st = run_block(xd, blob, kv, layer, batch, direct ? pos_dev : pd, direct ? y_dev : yd, ws, s, nullptr);
  if (st != FUTR_OK) return st;
  if (!direct && cudaMemcpyAsync(y_host, yd, xb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return FUTR_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(s));
}

futr_status futr_decode_step(const int32_t* tokens, const uint16_t* embedding, int32_t vocab,
                             const void* const* blobs, int32_t n_layers, const futr_kv* kv, int32_t batch,
                             const int32_t* pos, const float* g_final, const uint16_t* lm_head, float* logits,
                             const futr_ws* ws, void* stream) {
  if (!tokens || !embedding || !blobs || !pos || !g_final || !lm_head || !logits) return FUTR_ERR_INVALID_ARG;
  if (vocab <= 0 || vocab % 64) return FUTR_ERR_UNSUPPORTED;
  if (n_layers < 1 || !kv_ok(kv) || n_layers > kv->n_layers) return FUTR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(embedding) & 15) || (reinterpret_cast<uintptr_t>(lm_head) & 15))
    return FUTR_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const futr_status st = check_decode(blobs[l], kv, l, batch, ws);
    if (st != FUTR_OK) return st;
  }
  const futr_shape& s = ws->shape;
  const cudaStream_t st = as_stream(stream);
  void* base = ws->base;
  int* err = at<int>(base, ws->off_err);
  // the two staging rows of the workspace carry the residual stream from block
  // to block; h holds the LM head's activation and q' the norm factors
  uint16_t* buf[2] = {at<uint16_t>(base, ws->off_xin), at<uint16_t>(base, ws->off_yout)};
  uint16_t* xg = at<uint16_t>(base, ws->off_h);
  float* r = at<float>(base, ws->off_qrot);
  Range range("futr.step");
  if (launch_embed(tokens, embedding, vocab, s.hidden, batch, buf[0], err, st, true) != cudaSuccess)
    return FUTR_ERR_CUDA;
  for (int l = 0; l < n_layers; ++l) {
    const futr_status e = run_block(buf[l & 1], blobs[l], kv, l, batch, pos, buf[(l + 1) & 1], ws, st, nullptr);
    if (e != FUTR_OK) return e;
  }
  if (launch_final_norm(buf[n_layers & 1], g_final, s.hidden, s.rms_eps, batch, xg, r, st, true) != cudaSuccess)
    return FUTR_ERR_CUDA;
  return cuda_status(launch_lm_head(xg, lm_head, vocab, s.hidden, batch, r, logits, err, st, true));
}

futr_status futr_check(const futr_ws* ws, const futr_kv* kv, void* stream) {
  cudaStream_t s = as_stream(stream);
  // the guard words after every region (a write past a region's end)
  uint64_t g[kMaxGuards];
  if (ws_ok(ws) && check_guards(ws->base, g, ws_guards(*ws, g), at<int>(ws->base, ws->off_err), s) != cudaSuccess)
    return FUTR_ERR_CUDA;
  if (kv_ok(kv) && check_guards(kv->base, g, kv_guards(*kv, g), at<int>(kv->base, kv->err_offset), s) != cudaSuccess)
    return FUTR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FUTR_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return FUTR_ERR_CUDA;
  futr_status result = FUTR_OK;
  // error regions: word 0 the first error code, word 1 the abort word of the
  // bounded waits
  int* words[2] = {ws_ok(ws) ? at<int>(ws->base, ws->off_err) : nullptr,
                   kv_ok(kv) ? at<int>(kv->base, kv->err_offset) : nullptr};
  for (int i = 0; i < 2; ++i) {
    if (!words[i]) continue;
    int v[2] = {0, 0};
    if (cudaMemcpy(v, words[i], sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FUTR_ERR_CUDA;
    if (v[0] != 0 || v[1] != 0) {
      if (result == FUTR_OK) result = v[0] != 0 ? v[0] : FUTR_ERR_TIMEOUT;
      if (cudaMemset(words[i], 0, 16) != cudaSuccess) return FUTR_ERR_CUDA;
      // a launch that gave up on a wait left its split-K arrival counters (and
      // the persistent kernel's flags) mid-count: start them from zero again
      if (i == 0 && (v[0] == FUTR_ERR_TIMEOUT || v[1] != 0) && ws->cnt_words > 0 &&
          cudaMemset(at<uint8_t>(ws->base, ws->off_cnt), 0, ws->cnt_words * 4) != cudaSuccess)
        return FUTR_ERR_CUDA;
    }
  }
  return result;
}

}  // extern "C"

// Helpers for entry points defined in other files of the library.
namespace futr {
namespace host {

uint64_t workspace_bytes(const futr_shape& s, int max_batch, int capacity, int n_sm) {
  return ws_layout(s, max_batch, round16(capacity), n_sm).total;
}

// Describe a workspace of `bytes` at device address `base` without touching it.
void describe_workspace(const futr_shape& s, int max_batch, int capacity, int n_sm, void* base, futr_ws* d) {
  const int cap = round16(capacity);
  const WsLayout L = ws_layout(s, max_batch, cap, n_sm);
  *d = futr_ws{};
  d->shape = s;
  d->max_batch = max_batch;
  d->capacity = cap;
  d->n_sm = n_sm;
  d->base = base;
  d->bytes = L.total;
  d->off_err = L.err;
  d->off_qrot = L.qrot;
  d->off_o = L.o;
  d->off_h = L.h;
  d->off_a = L.a;
  d->off_xin = L.xin;
  d->off_yout = L.yout;
  d->off_pos = L.pos;
  d->off_part = L.part;
  d->part_bytes = L.part_bytes;
  d->off_apart = L.apart;
  d->apart_bytes = L.apart_bytes;
  d->off_cnt = L.cnt;
  d->cnt_words = L.cnt_words;
  d->magic = kWsMagic;
}

int sm_count() { return current_sm_count(); }

bool kv_valid(const futr_kv* kv) { return kv_ok(kv) && shape_ok(&kv->shape) && kv->capacity > 0; }

futr_status check_decode_args(const void* blob, const futr_kv* kv, int layer, int batch, const futr_ws* ws) {
  return check_decode(blob, kv, layer, batch, ws);
}

futr_status launch_block(const uint16_t* x, const void* blob, const futr_kv* kv, int layer, int batch,
                         const int32_t* pos, uint16_t* y, const futr_ws* ws, cudaStream_t st) {
  return run_block(x, blob, kv, layer, batch, pos, y, ws, st, nullptr);
}

}  // namespace host
}  // namespace futr
