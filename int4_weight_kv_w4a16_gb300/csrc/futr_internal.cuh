// Internal definitions shared by the libfutr kernels: packed layouts, PTX
// wrappers (mbarrier, bulk async copy, programmatic dependent launch,
// mma.sync, ldmatrix) and the fp32 rotation + INT4 quantizer used by both KV
// writers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "futr.h"

namespace futr {

// Occupancy answers (CTAs per SM, cluster sizes) decide the launch plans, and
// a workspace is sized from those plans: the first answer for a key is kept
// for the life of the process, so later plans always match the workspace.
// One table per call site (each passes its own lambda type).
template <class Query>
inline int remembered(uint64_t key, Query q) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> memo;
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  const int v = q();
  std::lock_guard<std::mutex> g(mu);
  return memo.emplace(key, v).first->second;
}

// One-time per-device set-up (kernel attributes): one bit per device, set
// atomically, because host threads may launch on several devices at once.
// Devices past 63 are set up on every call.
struct DeviceOnce {
  std::atomic<uint64_t> bits{0};
  bool done(int dev) const { return dev >= 0 && dev < 64 && (bits.load(std::memory_order_acquire) >> dev) & 1u; }
  void mark(int dev) {
    if (dev >= 0 && dev < 64) bits.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
};

inline uint64_t occ_key(int dev, int a, int b, size_t smem) {
  return ((uint64_t)(dev & 0xFF) << 56) | ((uint64_t)(a & 0xFF) << 48) | ((uint64_t)(b & 0xFF) << 40) |
         ((uint64_t)smem & 0xFFFFFFFFFFull);
}

// ----------------------------------------------------------------- layouts --
// Packed weights: a projection with N output rows and K inputs is cut into
// units of 128 rows x 128 inputs (one scale group).  Unit (rb, g) sits at
// byte ((rb * K/128) + g) * kUnitBytes of its section:
//   8 row tiles of 16 rows, each [half 0..1][lane 0..31][16 bytes]:
//     lane = 4*gr + t holds, for the k-steps ks = 4*half + j (j = word 0..3),
//     one 32-bit word with the 8 nibbles (code + 8) of rows gr, gr+8 and
//     columns 16ks + {2t, 2t+1, 2t+8, 2t+9}: nibble i (bits 4i..4i+3) is the
//     low half of register a_i, nibble i+4 its high half, where a0 = (gr, 2t),
//     a1 = (gr+8, 2t), a2 = (gr, 2t+8), a3 = (gr+8, 2t+8) -- the m16n8k16 A
//     fragment of that lane.
//   then 128 fp16 scales, one per row of the unit.
constexpr int kRowsPerBlock = 128;
constexpr int kGroup = 128;
constexpr int kUnitCodeBytes = kRowsPerBlock * kGroup / 2;   // 8192
constexpr int kUnitBytes = kUnitCodeBytes + kRowsPerBlock * 2; // 8448
constexpr int kHeaderBytes = 256;
constexpr uint64_t kBlobMagic = 0x3141345754554631ull;         // "1FUTW4A1"
constexpr uint64_t kKvMagic = 0x31564b3452545546ull;
constexpr uint64_t kWsMagic = 0x3153573452545546ull;
constexpr int kMaxBatch = 32;
constexpr int kMaxCapacity = 65536;  // positions per sequence

// KV stream of one (layer, seq, kv-head), capacity C (multiple of 16):
//   K codes: C/8 tiles of 8 positions x d/2 bytes; in a tile, lane 4*p + t
//     (p = position in tile) owns d/8 bytes = d/32 words; word j holds the
//     nibbles of dims 32j + {2t, 2t+8, 16+2t, 16+2t+8} in slots 0..3 and
//     dims 32j + {2t+1, 2t+9, 16+2t+1, 16+2t+9} in slots 4..7: slots (i, i+4)
//     form the fp16x2 register of the B fragment (k = dims, n = positions).
//   V codes: C/16 tiles of 16 positions x d/2 bytes; lane 4*gr + t owns d/4
//     bytes = d/16 words; word j holds dims 16j + gr (slots 0,1,4,5) and
//     16j + 8 + gr (slots 2,3,6,7) at tile positions 2t (slot 0/2), 2t+8
//     (1/3), 2t+1 (4/6), 2t+9 (5/7): the B fragment with k = positions,
//     n = dims.
//   K scales fp16 [C], V scales fp16 [C].
__host__ __device__ inline uint64_t kv_stream_bytes(int cap, int d) {
  return (uint64_t)cap * (uint64_t)(d + 4);
}

struct BlobSections {
  uint64_t off[4];   // QKV, O, GU, DOWN
  int rows[4];
  int cols[4];
  uint64_t total;
};

__host__ inline BlobSections blob_sections(const futr_shape& s) {
  BlobSections b;
  const int qkv = (s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim;
  b.rows[0] = qkv;          b.cols[0] = s.hidden;
  b.rows[1] = s.hidden;     b.cols[1] = s.n_q_heads * s.head_dim;
  b.rows[2] = 2 * s.inter;  b.cols[2] = s.hidden;
  b.rows[3] = s.hidden;     b.cols[3] = s.inter;
  uint64_t off = kHeaderBytes;
  for (int i = 0; i < 4; ++i) {
    b.off[i] = off;
    off += (uint64_t)(b.rows[i] / kRowsPerBlock) * (uint64_t)(b.cols[i] / kGroup) * kUnitBytes;
    off = (off + 255) & ~uint64_t(255);
  }
  b.total = off;
  return b;
}

struct BlobHeader {
  uint64_t magic;
  int32_t version;
  int32_t _pad;
  futr_shape shape;
};

// ------------------------------------------------------------ PTX helpers --
// Bounded waits.  Every wait gives up after kWaitNs, or as soon as another CTA
// of the same launch has recorded a time-out: the error region holds the first
// error code in word 0 and an abort word in word 1, which record_timeout sets
// and every waiting loop polls, so one failure ends the whole launch within
// microseconds instead of each CTA waiting out its own deadline.
constexpr unsigned long long kWaitNs = 50000000ull;  // 50 ms

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Arrival on a grid-wide counter: release of everything this CTA wrote
// before the preceding CTA barrier, acquire of what earlier arrivals wrote.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase of `bar` with parity `parity` (for lanes that
// share a warp with another spinning lane).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// True once some CTA has recorded a time-out in the error region `err`.
__device__ __forceinline__ bool aborted(const int* err) {
  return err && *reinterpret_cast<const volatile int*>(err + 1) != 0;
}

// Wait for the phase of `bar` with parity `parity` until the %globaltimer
// `deadline` (ns) or until the launch was aborted (see aborted); returns false
// then (the caller records FUTR_ERR_TIMEOUT and stops waiting).
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, unsigned long long deadline,
                                                const int* err) {
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u && (global_ns() > deadline || aborted(err))) return false;
  }
}

// After a time-out: wait (bounded, not cut short by the abort word) until the
// copies of the last `ring` stages issued into a ring of `ring` full barriers
// have landed, so that no bulk copy still writes into this CTA's shared memory
// when it exits.  Stage i completes phase i / ring of barrier i % ring; the
// last `ring` stages are the latest phase of their barriers.
__device__ __forceinline__ void drain_ring(uint64_t* full, int ring, int issued) {
  const unsigned long long dl = global_ns() + kWaitNs;
  for (int i = issued > ring ? issued - ring : 0; i < issued; ++i)
    mbar_wait_until(&full[i % ring], (uint32_t)(i / ring) & 1u, dl, nullptr);
}

// Pull [src, src + bytes) into L2 (no completion, no destination).  src
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: no-ops when the kernel was launched without it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* smem_row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(smem_row)));
}

// The four bf16x2 registers of a word of offset-8 codes: register i holds the
// nibbles at bits 4i and 16 + 4i.  0x4300 | u is the bf16 value 128 + u, so
// subtracting 136 (bf16 0x4308) leaves u - 8 exactly.  Written as one PTX
// sequence (3 shifts, 4 lop3 "(a & b) | c", 4 bf16x2 subtracts): the
// compiler's own lowering of the C expression issues more integer-pipe work.
__device__ __forceinline__ void nib4_bf16x2(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b32 s1, s2, s3, t0, t1, t2, t3;\n\t"
      "shr.b32 s1, %4, 4;\n\tshr.b32 s2, %4, 8;\n\tshr.b32 s3, %4, 12;\n\t"
      "lop3.b32 t0, %4, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "lop3.b32 t1, s1, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "lop3.b32 t2, s2, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "lop3.b32 t3, s3, 0x000F000F, 0x43004300, 0xEA;\n\t"
      "sub.rn.bf16x2 %0, t0, %5;\n\tsub.rn.bf16x2 %1, t1, %5;\n\t"
      "sub.rn.bf16x2 %2, t2, %5;\n\tsub.rn.bf16x2 %3, t3, %5;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w), "r"(0x43084308u));
}

// All four fp16x2 registers of a word (slots (i, i+4), i = 0..3) with one
// shift: fp16 keeps 10 mantissa bits, so a nibble at bits 4-7 of a half is
// exact too: 0x6400 | u << 4 is 1024 + 16u, and (1024 + 16u) / 16 - 72 = u - 8.
__device__ __forceinline__ void nib4_f16x2(uint32_t w, uint32_t (&r)[4]) {
  // one shift, 4 lop3, then 1032 subtracted (fp16 0x6408) or x / 16 - 72
  // (fp16 0x2C00, 0xD480)
  asm("{\n\t.reg .b32 s8, t0, t1, t2, t3;\n\t"
      "shr.b32 s8, %4, 8;\n\t"
      "lop3.b32 t0, %4, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 t1, %4, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "lop3.b32 t2, s8, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 t3, s8, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "sub.rn.f16x2 %0, t0, %5;\n\tfma.rn.f16x2 %1, t1, %6, %7;\n\t"
      "sub.rn.f16x2 %2, t2, %5;\n\tfma.rn.f16x2 %3, t3, %6, %7;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w), "r"(0x64086408u), "r"(0x2C002C00u), "r"(0xD480D480u));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// v0, v1 -> fp16x2 hi = (fp16(v0), fp16(v1)) and lo = fp16 of the remainders.
// Transpose of an 8x8 16-bit matrix held as a warp fragment (thread i:
// row i / 4, columns 2 (i % 4) and 2 (i % 4) + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ void split_half2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(v0, v1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// A bounded wait ran out: record the code and raise the abort word that every
// other wait of the launch polls.
__device__ __forceinline__ void record_timeout(int* err) {
  if (!err) return;
  atomicCAS(err, 0, FUTR_ERR_TIMEOUT);
  atomicExch(err + 1, 1);
}

// Debug build (compiled with -DFUTR_DEBUG): FUTR_DCHECK(cond, err) tests an
// index or range before a global access; a failed check records
// FUTR_ERR_BOUNDS with the source line (error word 2), raises the abort word
// so every bounded wait of the launch ends, and is false, so the caller skips
// the access.  In the release build it is the constant true and the condition
// is not evaluated.
__device__ __noinline__ inline bool dcheck_fail(int* err, int line) {
  if (err) {
    if (atomicCAS(err, 0, FUTR_ERR_BOUNDS) == 0) err[2] = line;
    atomicExch(err + 1, 1);
  }
  return false;
}
#ifdef FUTR_DEBUG
#define FUTR_DCHECK(cond, err) ((cond) ? true : ::futr::dcheck_fail((err), __LINE__))
#else
#define FUTR_DCHECK(cond, err) true
#endif

// ------------------------------------------------- rotation + quantizer --
// One warp holds a d-vector (d = 32*J, element i = lane + 32*j in v[j]).
// fp32 fast Walsh-Hadamard transform in blocks of nh (power of two <= d):
// stage s pairs i (bit s clear) with i + 2^s -> (a + b, a - b), ascending s;
// then one multiply by c = fp32(1/sqrt(nh)).
template <int J>
__device__ __forceinline__ void warp_fwht(float (&v)[J], int nh, float c) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
    if (h < nh) {
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float p = __shfl_xor_sync(0xffffffffu, v[j], h);
        v[j] = (lane & h) ? __fsub_rn(p, v[j]) : __fadd_rn(v[j], p);
      }
    }
  }
#pragma unroll
  for (int hj = 1; hj < J; hj <<= 1) {
    if (32 * hj < nh) {
#pragma unroll
      for (int j = 0; j < J; ++j) {
        if ((j & hj) == 0) {
          const float a = v[j], b = v[j + hj];
          v[j] = __fadd_rn(a, b);
          v[j + hj] = __fsub_rn(a, b);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < J; ++j) v[j] = __fmul_rn(v[j], c);
}

// INT4 round-to-nearest of a warp-held vector: s = fp16(max|v| / 7) (fp32
// division, saturating at 65504), code = clamp(rint(v / s), -8, 7), 0 if s == 0.
template <int J>
__device__ __forceinline__ __half warp_quant(const float (&v)[J], int (&code)[J]) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < J; ++j) m = fmaxf(m, fabsf(v[j]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const __half s = __float2half_rn(fminf(__fdiv_rn(m, 7.0f), 65504.0f));
  const float sf = __half2float(s);
#pragma unroll
  for (int j = 0; j < J; ++j) {
    int c = 0;
    if (sf > 0.f) {
      c = __float2int_rn(__fdiv_rn(v[j], sf));
      c = c < -8 ? -8 : (c > 7 ? 7 : c);
    }
    code[j] = c;
  }
  return s;
}

// Device view of one layer of the KV cache.
struct KvView {
  uint8_t* base;            // stream (layer, seq 0, kvh 0)
  uint64_t stream_bytes;
  int cap, d, n_kv;
  __device__ __forceinline__ uint8_t* stream(int seq, int kvh) const {
    return base + ((uint64_t)seq * n_kv + kvh) * stream_bytes;
  }
};

// Key word w (< d/8) of one position: the 8 codes of dims 32 j + 2 t + {0, 8,
// 16, 24, 1, 9, 17, 25} (t = w / (d/32), j = w % (d/32)) as nibbles code + 8.
// codes: the position's d codes (int8, dim order).
template <int d>
__device__ __forceinline__ uint32_t k_token_word(const int8_t* codes, int w) {
  const int t = w / (d / 32), j = w % (d / 32);
  const int base = 32 * j + 2 * t;
  const int dims[8] = {base, base + 8, base + 16, base + 24, base + 1, base + 9, base + 17, base + 25};
  uint32_t v = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) v |= (uint32_t)((codes[dims[i]] + 8) & 0xF) << (4 * i);
  return v;
}

// Value word w (< 8 d/16) of the 16-position tile holding position p: its
// word offset in the tile, the mask of position p's two nibbles in it and
// their new bits (dims 16 j + gr and 16 j + 8 + gr; gr = w / (d/16), j = w %
// (d/16)).
struct VWord {
  int off;
  uint32_t mask, bits;
};
template <int d>
__device__ __forceinline__ VWord v_token_word(const int8_t* codes, int p, int w) {
  const int p16 = p & 15;
  const int t = (p16 & 7) >> 1, hi = p16 >> 3, odd = p16 & 1;
  const int sh = 16 * odd + 4 * hi;
  const int gr = w / (d / 16), j = w % (d / 16);
  const uint32_t n0 = (uint32_t)((codes[16 * j + gr] + 8) & 0xF);
  const uint32_t n1 = (uint32_t)((codes[16 * j + 8 + gr] + 8) & 0xF);
  return VWord{(4 * gr + t) * (d / 16) + j, (0xFu << sh) | (0xFu << (sh + 8)), (n0 << sh) | (n1 << (sh + 8))};
}

// Write one token of one kv-head into slot p of a stream (one warp): codes
// (d int8 in [-8, 7], dim order, in shared memory) and scale.  K slots are
// plain stores of whole words; V slots update the nibbles of position p only
// (an atomic AND then an atomic OR per word), so other positions of the tile
// are left untouched.
template <int d>
__device__ __forceinline__ void put_k_token(uint8_t* strm, int cap, int p, const int8_t* codes, __half s) {
  const int lane = threadIdx.x & 31;
  // d/8 words per position, contiguous
  if (lane < d / 8) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(strm + (uint64_t)(p >> 3) * (4 * d) + (p & 7) * (d / 2));
    dst[lane] = k_token_word<d>(codes, lane);
  }
  if (lane == 0) {
    __half* ks = reinterpret_cast<__half*>(strm + (uint64_t)cap * d);
    ks[p] = s;
  }
}

template <int d>
__device__ __forceinline__ void put_v_token(uint8_t* strm, int cap, int p, const int8_t* codes, __half s) {
  const int lane = threadIdx.x & 31;
  uint32_t* tile = reinterpret_cast<uint32_t*>(strm + (uint64_t)cap * (d / 2) + (uint64_t)(p >> 4) * (8 * d));
  for (int w = lane; w < 8 * (d / 16); w += 32) {
    const VWord vw = v_token_word<d>(codes, p, w);
    // clear, then set, the nibbles of position p: two reductions on the word
    // (same thread, same address: applied in program order), no read back
    atomicAnd(tile + vw.off, ~vw.mask);
    atomicOr(tile + vw.off, vw.bits);
  }
  if (lane == 0) {
    __half* vs = reinterpret_cast<__half*>(strm + (uint64_t)cap * d + 2ull * cap);
    vs[p] = s;
  }
}

// The same from warp-held codes (code[j] of dim lane + 32 j); `scratch`: a
// per-warp shared buffer of d bytes.
template <int J>
__device__ __forceinline__ void store_k_token(uint8_t* strm, int cap, int p, const int (&code)[J],
                                              __half s, int8_t* scratch) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < J; ++j) scratch[lane + 32 * j] = (int8_t)code[j];
  __syncwarp();
  put_k_token<32 * J>(strm, cap, p, scratch, s);
  __syncwarp();
}

template <int J>
__device__ __forceinline__ void store_v_token(uint8_t* strm, int cap, int p, const int (&code)[J],
                                              __half s, int8_t* scratch) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < J; ++j) scratch[lane + 32 * j] = (int8_t)code[j];
  __syncwarp();
  put_v_token<32 * J>(strm, cap, p, scratch, s);
  __syncwarp();
}

// ------------------------------------------------------- host launchers --
cudaError_t launch_pack(const futr_shape& s, const float* wq, const float* wk, const float* wv,
                        const float* wo, const float* wg, const float* wu, const float* wd,
                        const float* ga, const float* gm, uint8_t* blob, cudaStream_t st);
cudaError_t launch_unpack(const futr_shape& s, const uint8_t* blob, int which, int8_t* codes,
                          uint16_t* scales, cudaStream_t st);
size_t gptq_scratch_bytes(const futr_shape& s);
// Synchronizes st; *bad_host = 1 when a dampened Hessian was not positive definite.
cudaError_t launch_pack_gptq(const futr_shape& s, const float* wq, const float* wk, const float* wv,
                             const float* wo, const float* wg, const float* wu, const float* wd, const float* ga,
                             const float* gm, const double* h_attn, const double* h_o, const double* h_mlp,
                             const double* h_down, double damp, void* scratch, uint8_t* blob, int* bad_host,
                             cudaStream_t st);
cudaError_t launch_rope_table(float2* table, int cap, int d, float theta, cudaStream_t st);
cudaError_t launch_kv_append(const futr_kv& kv, int layer, int seq0, int batch, const int* pos,
                             int n_tok, const uint16_t* k, const uint16_t* v, int* err,
                             cudaStream_t st);
cudaError_t launch_kv_read(const futr_kv& kv, int layer, int seq, int n_pos, int8_t* kc, uint16_t* ks,
                           int8_t* vc, uint16_t* vs, cudaStream_t st);
KvView kv_layer_view(const futr_kv& kv, int layer);
cudaError_t launch_embed(const int* tokens, const uint16_t* table, int vocab, int H, int batch, uint16_t* x,
                         int* err, cudaStream_t st, bool pdl);
cudaError_t launch_final_norm(const uint16_t* y, const float* g, int H, float eps, int batch, uint16_t* xg, float* r,
                              cudaStream_t st, bool pdl);
cudaError_t launch_lm_head(const uint16_t* xg, const uint16_t* w, int vocab, int H, int batch, const float* r,
                           float* logits, int* err, cudaStream_t st, bool pdl);

}  // namespace futr
