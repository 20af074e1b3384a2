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
//     receives (mbarrier completion) the weight unit (codes + scales, 8448 B)
//     by a 1-D bulk copy and the matching activation tile by one 2-D tensor
//     copy: a box of 136 inputs x batch rows lands as rows of 272 bytes (128
//     inputs + 8 that keep ldmatrix free of bank conflicts; inputs past K read
//     as zero).  A single row (batch 1) comes by a 256-byte bulk copy, which
//     measured faster than the tensor copy there.  Weight units of the first stages are
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
// Batch 17..32 of the residual and SwiGLU projections runs a variant with the
// same stream, unpacking and epilogue on the 5th-generation tensor cores
// (tcgen05.mma with A in tensor memory; proj_tc_kernel below).
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "futr_internal.cuh"
#include "proj.cuh"
#include "proj_dev.cuh"

namespace futr {

namespace {

// ------------------------------------------------ cluster split-K tail --
// The S CTAs of a row block form one thread-block cluster (cluster rank =
// split index).  After its K-range each CTA leaves its partial tile [batch row]
// [128 rows] and its sums of squares in its own shared memory; a cluster
// barrier; then every CTA adds, for the outputs it owns, the S partials in
// split order (distributed-shared-memory loads, all S in flight) and runs the
// fused epilogue on them:
//   RESID : rows [r*128/S, (r+1)*128/S) of the block, every batch row
//   SWIGLU: outputs [r*64/S, (r+1)*64/S) (gate row j, up row 64 + j)
//   QKV   : head tasks (batch row, head) r, r + S, ... (one warp each)
// A second cluster barrier keeps every CTA's shared memory alive until the
// others have read it.  Every thread of every CTA (the producer warp
// included) reaches both barriers exactly once; a time-out anywhere in the
// cluster is visible through the abort word after the first one, and then no
// output is written.  No global partial records, counters or atomics.
constexpr int kMaxProjCluster = 16;

__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// The second barrier publishes nothing: every value this CTA read from the
// others' shared memory has been consumed by the stores before it (so those
// loads have completed), so its arrival needs no release.  (The debug build,
// whose failed checks skip stores and leave loaded values unused, keeps the
// release.)
__device__ __forceinline__ void cl_arrive_relaxed() {
#ifdef FUTR_DEBUG
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
#else
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
#endif
}

// Shared-memory address of `local` in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cl_map(const void* local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

__device__ __forceinline__ float cl_ld(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// sum over the cluster's S CTAs, in rank order from 0, of the float at `local`
// (eight loads in flight per round)
__device__ __forceinline__ float cl_sum(const float* local, int S) {
  float acc = 0.f;
  for (int s0 = 0; s0 < S; s0 += 8) {
    float v[8];
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s0 + s < S) v[s] = cl_ld(cl_map(local, s0 + s));
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s0 + s < S) acc += v[s];
  }
  return acc;
}

// The owned outputs of this CTA (rank `rank` of the cluster of row block rb),
// from the S partial tiles `red` and sums of squares `ss`.  Consumer threads.
template <int EPI>
__device__ __forceinline__ void cluster_epilogue(const ProjArgs& a, const float* red, const float* ss, int rb,
                                                 int S, int rank) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (EPI == kEpiResid) {
    const int r0 = rank * kRowsPerBlock / S, nr = (rank + 1) * kRowsPerBlock / S - r0;
    for (int e = tid; e < nr * a.batch; e += kCW * 32) {
      const int n = e / nr, row = r0 + (e - n * nr);
      const size_t o = (size_t)n * a.out_ld + (size_t)rb * kRowsPerBlock + row;
      const float res = __bfloat162float(__ldcg(a.resid + o));
      const float v = cl_sum(red + n * kRedLd + row, S);
      if (FUTR_DCHECK(o < a.out_cap, a.err)) a.out[o] = __float2bfloat16_rn(res + v);
    }
  } else if (EPI == kEpiSwiglu) {
    const int j0 = rank * 64 / S, nj = (rank + 1) * 64 / S - j0;
    for (int e = tid; e < nj * a.batch; e += kCW * 32) {
      const int n = e / nj, j = j0 + (e - n * nj);
      const float g0 = cl_sum(red + n * kRedLd + j, S);
      const float u0 = cl_sum(red + n * kRedLd + 64 + j, S);
      const float sq = cl_sum(ss + n, S);
      const float rn = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(sq, (float)a.K) + a.eps));
      const float g = rn * g0;
      const float u = rn * u0;
      const float sg = __fdiv_rn(g, 1.0f + expf(-g));
      const size_t o = (size_t)n * a.out_ld + (size_t)rb * 64 + j;
      if (FUTR_DCHECK(o < a.out_cap, a.err)) a.out[o] = __float2bfloat16_rn(sg * u);
    }
  } else {
    if (rb == 0 && rank == 0 && tid == 0 && a.blob_magic && *a.blob_magic != kBlobMagic)
      set_err(a.err, FUTR_ERR_BAD_BLOB);
    const int hpr = kRowsPerBlock / a.d, ntask = a.batch * hpr;
    for (int task = rank + S * warp; task < ntask; task += S * kCW) {
      const int n = task / hpr, hl = task - n * hpr, hg = rb * hpr + hl;
      const HeadPre hp = head_pre(a, n, hg);
      const float sq = cl_sum(ss + n, S);
      const float rn = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(sq, (float)a.K) + a.eps));
      if (a.d == 128) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = cl_sum(red + n * kRedLd + hl * 128 + lane + 32 * j, S) * rn;
        qkv_head_core<4>(a, v, n, hg, hp);
      } else {
        float v[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) v[j] = cl_sum(red + n * kRedLd + hl * 64 + lane + 32 * j, S) * rn;
        qkv_head_core<2>(a, v, n, hg, hp);
      }
    }
  }
}

// Which instantiations reduce inside a cluster (see cluster_epilogue and the
// planner); the others through global split records added by the last CTA of
// the row block.
template <int NTP, int EPI>
constexpr bool cluster_reduce() {
  return NTP != 0 && EPI != kEpiSwiglu && EPI != kEpiQkvRec;
}

// NTP: batch tiles of 8 columns, 1..4; 0 = one batch row (one tile, the
// activation row by a bulk copy)

template <int NTP, int EPI>
__device__ __forceinline__ void proj_body(const ProjArgs& a, const CUtensorMap* xmap) {
  constexpr int NT = NTP == 0 ? 1 : NTP;
  constexpr bool kRow1 = NTP == 0;
  constexpr bool kCluster = cluster_reduce<NTP, EPI>();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // tensor copies want a 128-byte aligned destination: the base is rounded up
  // (one row takes only 16-byte aligned bulk copies and uses it as it is)
  uint8_t* smem = kRow1 ? smem_raw
                        : reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
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

  if (tid == 0) {
    flag[0] = 0;
    flag[1] = 0;
    flag[2] = 0;
    flag[3] = 0;
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
      const uint32_t tx = kUnitBytes + (kRow1 ? kGroup * 2 : (uint32_t)a.batch * kTileLd * 2);
      // test hook: no copy is issued; debug build: the units lie in the section
      const bool hold = (a.withhold && blockIdx.x == 0) || !FUTR_DCHECK(rb < a.n_rb && g1 <= a.n_groups, a.err);
      const int pre = hold ? 0 : (ng < R ? ng : R);
      if (!kRow1) prefetch_map(xmap);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], tx);
        bulk_g2s(stages + (size_t)i * a.stage_bytes, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[i]);
      }
      pdl_wait();  // the activations come from the previous kernel
      const unsigned long long deadline = global_ns() + kWaitNs;
      for (int i = 0; i < pre; ++i) issue_tile<kRow1>(a, xmap, stages + (size_t)i * a.stage_bytes, g0 + i, &full[i]);
      int slot = 0, issued = pre;
      uint32_t phase = 0;
      for (int i = hold ? ng : R; i < ng; ++i) {
        if (!mbar_wait_until(&empty[slot], phase, deadline, a.err)) {
          record_timeout(a.err);
          break;
        }
        uint8_t* st = stages + (size_t)slot * a.stage_bytes;
        mbar_arrive_expect_tx(&full[slot], tx);
        bulk_g2s(st, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[slot]);
        issue_tile<kRow1>(a, xmap, st, g0 + i, &full[slot]);
        issued = i + 1;
        if (++slot == R) {
          slot = 0;
          phase ^= 1u;
        }
      }
      publish_issued(flag, issued);
      // QKV whose epilogue runs in the attention kernel: the blob header check
      if (EPI == kEpiQkvRec && blockIdx.x == 0 && a.blob_magic && *a.blob_magic != kBlobMagic)
        set_err(a.err, FUTR_ERR_BAD_BLOB);
    } else {
      pdl_wait();
    }
    if (kCluster) {
      // the cluster's two barriers (see cluster_epilogue)
      cl_arrive();
      cl_wait();
      cl_arrive_relaxed();
      cl_wait();
    }
    return;
  }

  // ----------------------------------------------------------- consumers --
  pdl_wait();
  const unsigned long long deadline = global_ns() + kWaitNs;
  bool ok = true;
  // QKV with global records (batch 1): warp w's head task's position and RoPE
  // factors, loaded now and used by the epilogue (their latency hides under
  // the K-loop instead of lengthening the tail)
  HeadPre hp_pre{};
  if (EPI == kEpiQkv && !kCluster) {
    const int hpr = kRowsPerBlock / a.d;
    if (warp < a.batch * hpr) hp_pre = head_pre(a, warp / hpr, rb * hpr + warp % hpr);
  }

  float acc[kMT][NT][4];
#pragma unroll
  for (int m = 0; m < kMT; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][nt][e] = 0.f;

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
    if (!mbar_wait_until(&full[slot], phase, deadline, a.err)) {
      ok = false;
      break;
    }
    unit_mma<NT, EPI != kEpiResid>(stages + (size_t)slot * a.stage_bytes, xrow, sq_off, a.batch, acc, ssq);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the stage
    if (++slot == R) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (EPI != kEpiResid) ssq_to_smem<NT>(ssq, ss, a.batch);
  if (!kCluster) {
    // split records in global memory, the last CTA of the row block reduces
    // (accumulator fragments -> epilogue tile in the ring, which every warp
    // has left by then)
    proj_tail<NT, EPI>(a, reinterpret_cast<float*>(smem), rb, a.S, sk, ss, flag, ok,
                       [&](float* red) { acc_to_red<NT>(acc, red); }, []() {},
                       EPI == kEpiQkv ? &hp_pre : nullptr);
    if (flag[1] && tid == 0) drain_after_timeout(smem, a.off_misc, a.ring);
    return;
  }
  if (!ok) record_timeout(a.err);  // before the cluster barrier: the others see the abort word after it
  // accumulator fragments -> partial tile [batch row][block row] (the ring,
  // which every warp has left by then)
  consumer_sync();
  float* red = reinterpret_cast<float*>(smem);
  acc_to_red<NT>(acc, red);
  cl_arrive();  // this CTA's partial tile and sums of squares are complete
  cl_wait();
  const bool live = !aborted(a.err);
  if (live) cluster_epilogue<EPI>(a, red, ss, rb, a.S, sk);
  cl_arrive_relaxed();  // done reading the other CTAs' shared memory
  cl_wait();
  // after a time-out (here or in another CTA, which stops this CTA's waits
  // too), let this CTA's copies land before it exits
  if (!live && tid == 0) drain_after_timeout(smem, a.off_misc, a.ring);
}

// ------------------------------------------------- tensor-core variant --
// Batch 17..32: the same unit stream and epilogue, with the products on the
// 5th-generation tensor cores.  Per unit (128 rows x 128 inputs):
//   warps 0..3 unpack their 32 rows' codes into bf16 MMA fragments (the same
//     registers the mma.sync path feeds) and store them to tensor memory with
//     tcgen05.st.16x128b.x2, which lays a 16-row fragment of one k-step out as
//     16 lanes x 8 columns in natural k order: A = 128 lanes (rows) x 64
//     columns (bf16 pairs);
//   warps 5 and 6 (one thread each) issue the 8 tcgen05.mma kind::f16 (M 128,
//     N 32, K 16) of the even and the odd units: A from tensor memory, B = the
//     activation tile in shared memory (K-major, two boxes of 32 rows x 64
//     inputs written by 2-D tensor copies with the 128-byte swizzle, read
//     through a 128-byte-swizzle descriptor), D = fp32 in tensor memory,
//     then tcgen05.commit signals the consumers and frees the ring slot.  An
//     issuing thread is held ~60 ns per MMA whatever N is (measured), while
//     issuers in different warps overlap: two issuers halve the cost;
//   warps 0..3 read D back two units later (tcgen05.ld.32x32b: thread = row,
//     32 batch columns), multiply by the row's group scale and add into
//     registers.
// A has three buffers and D two (256 tensor-memory columns per CTA, two CTAs
// per SM), so the unpacking of unit i, the MMAs of units i - 1 and i - 2 and
// the read-back of unit i - 2 overlap.  Every wait is bounded; tensor memory
// is freed before the epilogue, once both issuers are past their last MMA
// (and, after a time-out, their last commits have landed).  Used for the
// residual and SwiGLU epilogues (see plan_projection).
constexpr int kTcCols = 256;                       // tensor-memory columns per CTA
constexpr int kTcA = 0;                            // A[b], b < 3: columns 64 b .. 64 b + 63
constexpr int kTcD = 192;                          // D[b], b < 2: columns 192 + 32 b .. + 31
constexpr int kTcTile = 32 * kGroup * 2;           // activation tile: 32 rows x 128 inputs, bf16
constexpr int kTcStage = 17 * 1024;                // tile (8 KB) + weight unit (8448 B), padded to 1 KB
constexpr int kTcThreads = (kCW + 3) * 32;         // consumers, producer, two MMA issuers
constexpr int kTcMisc = 32 * 4 + 16 + (2 * kMaxRing + 5) * 8 + 32;
// instruction descriptor: D f32, A and B bf16, both K-major, N = 32, M = 128
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory operand descriptor, K-major with the 128-byte swizzle: rows of
// 128 bytes in 8-row atoms of 1 KB (sbo = 1024); a k-step starts 32 bytes
// further along the row
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(kTcIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_st_frag(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x2.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

__device__ __forceinline__ void tc_ld_row32(uint32_t taddr, float (&v)[32]) {
  uint32_t u[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]),
        "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]),
        "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
        "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
}

// activation tile of group g: inputs 128 g .. 128 g + 127 as two 4 KB boxes
__device__ __forceinline__ void tc_issue_tile(uint8_t* dst, const CUtensorMap* map, int g, uint64_t* bar) {
  tma_2d_box(dst, map, kGroup * g, 0, bar);
  tma_2d_box(dst + 4096, map, kGroup * g + 64, 0, bar);
}

template <int EPI>
__global__ void __launch_bounds__(kTcThreads, 2)
    proj_tc_kernel(const __grid_constant__ ProjArgs a, const __grid_constant__ CUtensorMap xmap) {
  constexpr int NT = 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.x / a.S, sk = blockIdx.x - rb * a.S;
  const int g0 = (int)(((long long)sk * a.n_groups) / a.S);
  const int g1 = (int)(((long long)(sk + 1) * a.n_groups) / a.S);
  const int ng = g1 - g0, R = a.ring;

  uint8_t* stages = smem;
  float* ss = reinterpret_cast<float*>(smem + a.off_misc);  // [32] sum of squares per batch row
  int* flag = reinterpret_cast<int*>(ss + 32);                // [4]
  uint64_t* full = reinterpret_cast<uint64_t*>(flag + 4);
  uint64_t* empty = full + kMaxRing;   // released by the MMA commit of the slot's unit
  uint64_t* aready = empty + kMaxRing; // [3] the 4 consumer warps stored A[b] (and read D two units back)
  uint64_t* mdone = aready + 3;        // [2] the MMAs into D[b] (and their reads of A) completed
  uint32_t* tbase = reinterpret_cast<uint32_t*>(mdone + 2);
  int* last_issued = reinterpret_cast<int*>(tbase + 1);  // [2] per issuer
  int* issuers_done = last_issued + 2;

  if (tid == 0) {
    flag[0] = 0;
    flag[1] = 0;
    flag[2] = 0;
    flag[3] = 0;
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 3; ++b) mbar_init(&aready[b], kCW);
    for (int b = 0; b < 2; ++b) mbar_init(&mdone[b], 1);
    last_issued[0] = last_issued[1] = -1;
    *issuers_done = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tbase)),
                 "r"(kTcCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tbase;
  pdl_trigger();

  const uint8_t* unit0 = a.w + ((size_t)rb * a.n_groups + g0) * kUnitBytes;
  if (warp == kCW) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const uint32_t tx = kUnitBytes + kTcTile;
      const int pre = ng < R ? ng : R;
      prefetch_map(&xmap);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], tx);
        bulk_g2s(stages + (size_t)i * kTcStage + kTcTile, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[i]);
      }
      pdl_wait();  // the activations come from the previous kernel
      const unsigned long long deadline = global_ns() + kWaitNs;
      for (int i = 0; i < pre; ++i) tc_issue_tile(stages + (size_t)i * kTcStage, &xmap, g0 + i, &full[i]);
      int slot = 0, issued = pre;
      uint32_t phase = 0;
      for (int i = R; i < ng; ++i) {
        if (!mbar_wait_until(&empty[slot], phase, deadline, a.err)) {
          record_timeout(a.err);
          break;
        }
        uint8_t* st = stages + (size_t)slot * kTcStage;
        mbar_arrive_expect_tx(&full[slot], tx);
        bulk_g2s(st + kTcTile, unit0 + (size_t)i * kUnitBytes, kUnitBytes, &full[slot]);
        tc_issue_tile(st, &xmap, g0 + i, &full[slot]);
        issued = i + 1;
        if (++slot == R) {
          slot = 0;
          phase ^= 1u;
        }
      }
      publish_issued(flag, issued);
    } else {
      pdl_wait();
    }
    return;
  }

  if (warp > kCW) {
    // ----------------------------------------------------- MMA issuers --
    // warp kCW + 1 + b issues units i = b, b + 2, ... into D[b]
    const int b = warp - kCW - 1;
    if (lane == 0) {
      const unsigned long long deadline = global_ns() + kWaitNs;
      bool ok = true;
      for (int i = b; i < ng; i += 2) {
        const int slot = i % R, ba = i % 3;
        // the tile has landed; the four consumer warps stored A(i) and read
        // D(i - 2), the previous contents of D[b]
        if (!mbar_wait_until(&full[slot], (uint32_t)(i / R) & 1u, deadline, a.err) ||
            !mbar_wait_until(&aready[ba], (uint32_t)(i / 3) & 1u, deadline, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tile = smem_u32(stages + (size_t)slot * kTcStage);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma(tm + kTcD + 32 * b, tm + kTcA + 64 * ba + 8 * ks,
                 tc_desc_sw128(tile + 4096 * (ks >> 2) + 32 * (ks & 3)), ks > 0);
        tc_commit(&mdone[b]);
        tc_commit(&empty[slot]);  // the ring slot is free once these MMAs have read the tile
        last_issued[b] = i;
      }
      if (!ok) {
        record_timeout(a.err);
        flag[1] = 1;
      }
      __threadfence_block();
      atomicAdd(issuers_done, 1);  // no MMA of this warp is issued after this point
    }
    return;
  }

  // ----------------------------------------------------------- consumers --
  pdl_wait();
  const unsigned long long deadline = global_ns() + kWaitNs;
  bool ok = true;
  float acc[32];
#pragma unroll
  for (int n = 0; n < 32; ++n) acc[n] = 0.f;
  // RMSNorm sum of squares: thread t squares one 16-byte chunk of tile row
  // n = t / 16 + 8p, box (t % 16) / 8, stored chunk t % 8 (which inputs the
  // chunk holds under the swizzle does not matter for the sum); bytes
  const int sq_off = ((tid & 15) >> 3) * 4096 + (tid >> 4) * 128 + (tid & 7) * 16;
  float ssq[NT];
#pragma unroll
  for (int p = 0; p < NT; ++p) ssq[p] = 0.f;
  const uint32_t lq = (uint32_t)(32 * warp) << 16;  // this warp's lane quarter
  const int row = 32 * warp + lane;                  // block row of this thread's D lane
  float s1 = 0.f, s2 = 0.f;  // group scales of units i - 1 and i - 2 for this row
  int slot = 0;
  uint32_t phase = 0;
  for (int i = 0; i < ng + 2; ++i) {
    float s0 = 0.f;
    if (i < ng) {
      const uint8_t* st = stages + (size_t)slot * kTcStage;
      const int ba = i % 3;
      if (!mbar_wait_until(&full[slot], phase, deadline, a.err)) {
        ok = false;
        break;
      }
      const uint4* wt = reinterpret_cast<const uint4*>(st + kTcTile + kMT * warp * 1024);
      s0 = __half2float(reinterpret_cast<const __half*>(st + kTcTile + kUnitCodeBytes)[row]);
      uint32_t words[kMT][8];
#pragma unroll
      for (int m = 0; m < kMT; ++m) {
        const uint4 w0 = wt[64 * m + lane], w1 = wt[64 * m + 32 + lane];
        words[m][0] = w0.x; words[m][1] = w0.y; words[m][2] = w0.z; words[m][3] = w0.w;
        words[m][4] = w1.x; words[m][5] = w1.y; words[m][6] = w1.z; words[m][7] = w1.w;
      }
      // A[ba] was last read by the MMAs of unit i - 3, whose completion this
      // warp waited for before reading D of that unit
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          uint32_t af[4];
          nib4_bf16x2(words[m][ks], af);
          tc_st_frag(tm + lq + ((uint32_t)(16 * m) << 16) + kTcA + 64 * ba + 8 * ks, af);
        }
      if (EPI != kEpiResid) {
#pragma unroll
        for (int p = 0; p < NT; ++p)
          if ((tid >> 4) + 8 * p < a.batch) {
            const uint4 v = *reinterpret_cast<const uint4*>(st + sq_off + 1024 * p);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = __uint_as_float(u[j] << 16), hi = __uint_as_float(u[j] & 0xffff0000u);
              ssq[p] = fmaf(lo, lo, fmaf(hi, hi, ssq[p]));
            }
          }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    if (i >= 2) {
      // D of unit i - 2; its buffer is overwritten by the MMAs of unit i,
      // which wait for this warp's arrival below
      const int v = i - 2, bd = v & 1;
      if (!mbar_wait_until(&mdone[bd], (uint32_t)(v >> 1) & 1u, deadline, a.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float d[32];
      tc_ld_row32(tm + lq + kTcD + 32 * bd, d);
#pragma unroll
      for (int n = 0; n < 32; ++n) acc[n] = fmaf(s2, d[n], acc[n]);
    }
    if (i < ng) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aready[i % 3]);  // A(i) stored, D(i - 2) read
      if (++slot == R) {
        slot = 0;
        phase ^= 1u;
      }
    }
    s2 = s1;
    s1 = s0;
  }
  if (!ok) {
    record_timeout(a.err);
    flag[1] = 1;
  }
  consumer_sync();
  if (warp == 0) {
    // tensor memory is freed once the last issued MMAs have landed (already
    // waited for on the normal path; bounded here for a path that timed out)
    // both issuers are past their last MMA (bounded wait); on the normal path
    // every MMA has completed already (all units' D were read back), after a
    // time-out the issuers' last commits are waited for
    if (lane == 0) {
      const unsigned long long dl = global_ns() + kWaitNs;
      while (*(volatile int*)issuers_done < 2 && global_ns() < dl) {
      }
      __threadfence_block();
    }
    __syncwarp();
    if (lane < 2 && flag[1]) {
      const int v = *(volatile int*)&last_issued[lane];
      if (v >= 0 && !mbar_wait_until(&mdone[lane], (uint32_t)(v >> 1) & 1u, global_ns() + kWaitNs, nullptr))
        record_timeout(a.err);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(kTcCols) : "memory");
  }
  if (EPI != kEpiResid) {
#pragma unroll
    for (int p = 0; p < NT; ++p) {
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) ssq[p] += __shfl_xor_sync(0xffffffffu, ssq[p], o);
      const int n = (tid >> 4) + 8 * p;
      if ((tid & 15) == 0 && n < a.batch) ss[n] = ssq[p];
    }
  }
  // thread t holds block row t for batch columns 0..31
  proj_tail<NT, EPI>(
      a, reinterpret_cast<float*>(smem), rb, a.S, sk, ss, flag, ok,
      [&](float* red) {
#pragma unroll
        for (int n = 0; n < 32; ++n) red[n * kRedLd + tid] = acc[n];
      },
      []() {});
  if (flag[1] && tid == 0) drain_after_timeout(smem, a.off_misc, a.ring);
}

template <int NT, int EPI>
__global__ void __launch_bounds__(kThreads, NT <= 1 ? 6 : 3) proj_kernel(const ProjArgs a, const __grid_constant__ CUtensorMap xmap) {
  proj_body<NT, EPI>(a, &xmap);
}

// Three or four batch tiles: at most 128 registers, so three CTAs share an SM.
template <int NT, int EPI>
__global__ void __maxnreg__(128) proj_kernel_wide(const ProjArgs a, const __grid_constant__ CUtensorMap xmap) {
  proj_body<NT, EPI>(a, &xmap);
}

template <int NT, int EPI>
constexpr void (*proj_entry())(ProjArgs, CUtensorMap) {
  if constexpr (NT >= 3)
    return proj_kernel_wide<NT, EPI>;
  else
    return proj_kernel<NT, EPI>;
}

template <int NT, int EPI>
cudaError_t configure(int dev) {
  static DeviceOnce configured;
  if (configured.done(dev)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(proj_entry<NT, EPI>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kProjMaxSmem);
  if (e != cudaSuccess) return e;
  // every kernel of the step asks for the maximum shared-memory carveout, so
  // CTAs of consecutive kernels can share an SM (programmatic overlap)
  e = cudaFuncSetAttribute(proj_entry<NT, EPI>(), cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // clusters of up to 16 CTAs (the split-K clusters)
  e = cudaFuncSetAttribute(proj_entry<NT, EPI>(), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  configured.mark(dev);
  return cudaSuccess;
}

template <int NT, int EPI>
cudaError_t launch_one(const ProjArgs& a, int grid, size_t smem, cudaStream_t st, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure<NT, EPI>(dev);
  if (e != cudaSuccess) return e;
  // with the cluster reduction the S CTAs of a row block are one cluster
  // (cluster_epilogue reads the shared memory of ranks 0..S-1, so the cluster
  // size must be exactly S)
  if (a.cluster != (cluster_reduce<NT, EPI>() ? 1 : 0)) return cudaErrorInvalidValue;  // fixed per instantiation
  if (a.cluster && (a.S < 1 || a.S > kMaxProjCluster || grid % a.S != 0)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (a.cluster) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)a.S;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  CUtensorMap xmap;
  if (NT == 0)
    memset(&xmap, 0, sizeof(xmap));  // one row: no tensor copy
  else if (!make_proj_tile_map(&xmap, a.xin, a.batch, a.K, a.batch))
    return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, proj_entry<NT, EPI>(), a, xmap);
}

template <int EPI>
cudaError_t launch_nt(int nt, const ProjArgs& a, int grid, size_t smem, cudaStream_t st, bool pdl) {
  switch (nt) {
    case 1: return a.batch == 1 ? launch_one<0, EPI>(a, grid, smem, st, pdl) : launch_one<1, EPI>(a, grid, smem, st, pdl);
    case 2: return launch_one<2, EPI>(a, grid, smem, st, pdl);
    case 3: return launch_one<3, EPI>(a, grid, smem, st, pdl);
    default: return launch_one<4, EPI>(a, grid, smem, st, pdl);
  }
}

template <int EPI>
cudaError_t configure_tc(int dev) {
  static DeviceOnce configured;
  if (configured.done(dev)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(proj_tc_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjMaxSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(proj_tc_kernel<EPI>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  configured.mark(dev);
  return cudaSuccess;
}

template <int EPI>
cudaError_t launch_tc(const ProjArgs& a, int grid, size_t smem, cudaStream_t st, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure_tc<EPI>(dev);
  if (e != cudaSuccess) return e;
  CUtensorMap xmap;
  if (!make_act_tile_map(&xmap, a.xin, a.batch, a.K)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, proj_tc_kernel<EPI>, a, xmap);
}

int resident_tc(int epi, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return remembered(occ_key(dev, 5, epi, smem), [&]() {
    int n = 0;
    cudaError_t e = cudaSuccess;
    if (epi == kEpiResid) {
      e = configure_tc<kEpiResid>(dev);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, proj_tc_kernel<kEpiResid>, kTcThreads, smem);
    } else {
      e = configure_tc<kEpiSwiglu>(dev);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, proj_tc_kernel<kEpiSwiglu>, kTcThreads, smem);
    }
    return e == cudaSuccess ? n : 0;
  });
}

int resident_ctas(int nt, int epi, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return remembered(occ_key(dev, nt, epi, smem), [&]() {
  int n = 0;
  cudaError_t e = cudaSuccess;
#define FUTR_OCC(NT_, EPI_)                                                               \
  if (nt == NT_ && epi == EPI_) {                                                         \
    e = configure<NT_, EPI_>(dev);                                                        \
    if (e == cudaSuccess)                                                                 \
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, proj_entry<NT_, EPI_>(), kThreads, smem); \
  }
  FUTR_OCC(0, 0) FUTR_OCC(1, 0) FUTR_OCC(2, 0) FUTR_OCC(3, 0) FUTR_OCC(4, 0)
  FUTR_OCC(0, 1) FUTR_OCC(1, 1) FUTR_OCC(2, 1) FUTR_OCC(3, 1) FUTR_OCC(4, 1)
  FUTR_OCC(0, 2) FUTR_OCC(1, 2) FUTR_OCC(2, 2) FUTR_OCC(3, 2) FUTR_OCC(4, 2)
  FUTR_OCC(0, 3) FUTR_OCC(1, 3) FUTR_OCC(2, 3) FUTR_OCC(3, 3) FUTR_OCC(4, 3)
#undef FUTR_OCC
  return e == cudaSuccess ? n : 0;
  });
}

// Largest split-K cluster the device schedules for this instantiation (at
// most kMaxProjCluster).
int max_proj_cluster(int nt, int epi, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  return remembered(occ_key(dev, 16 + nt, epi, smem), [&]() {
    int n = 0;
    cudaError_t e = cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMaxProjCluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
#define FUTR_CL(NT_, EPI_)                                                                   \
  if (nt == NT_ && epi == EPI_) {                                                            \
    e = configure<NT_, EPI_>(dev);                                                           \
    if (e == cudaSuccess) e = cudaOccupancyMaxPotentialClusterSize(&n, proj_entry<NT_, EPI_>(), &cfg); \
  }
    FUTR_CL(0, 0) FUTR_CL(1, 0) FUTR_CL(2, 0) FUTR_CL(3, 0) FUTR_CL(4, 0)
    FUTR_CL(0, 1) FUTR_CL(1, 1) FUTR_CL(2, 1) FUTR_CL(3, 1) FUTR_CL(4, 1)
    FUTR_CL(0, 2) FUTR_CL(1, 2) FUTR_CL(2, 2) FUTR_CL(3, 2) FUTR_CL(4, 2)
#undef FUTR_CL
    if (e != cudaSuccess || n < 1) {
      cudaGetLastError();
      return 1;
    }
    return n < kMaxProjCluster ? n : kMaxProjCluster;
  });
}

// Clusters of S CTAs of this instantiation that the device holds at once (a
// cluster sits within one GPC, so this can be fewer than the resident CTAs
// per SM x SMs / S).
int active_clusters(int nt, int epi, size_t smem, int S) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return remembered(occ_key(dev, 64 + nt * 16 + S - 1, epi, smem), [&]() {
    int n = 0;
    cudaError_t e = cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(S * 64));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#define FUTR_AC(NT_, EPI_)                                                              \
  if (nt == NT_ && epi == EPI_) {                                                       \
    e = configure<NT_, EPI_>(dev);                                                      \
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, proj_entry<NT_, EPI_>(), &cfg); \
  }
    FUTR_AC(1, 0) FUTR_AC(2, 0) FUTR_AC(3, 0) FUTR_AC(4, 0)
    FUTR_AC(1, 1) FUTR_AC(2, 1) FUTR_AC(3, 1) FUTR_AC(4, 1)
    FUTR_AC(1, 2) FUTR_AC(2, 2) FUTR_AC(3, 2) FUTR_AC(4, 2)
#undef FUTR_AC
    if (e != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  });
}

}  // namespace

ProjPlan plan_projection(int rows, int cols, int batch, int n_sm, int force_split, int epi) {
  ProjPlan p{};
  p.n_rb = rows / kRowsPerBlock;
  p.n_groups = cols / kGroup;
  p.nt = (batch + 7) / 8;
  p.epi = epi;
  // batch 17..32: the tensor-core kernel (32 batch columns, two CTAs per SM)
  // for the projections where it measured faster than mma.sync at batch 32
  // on the 8B and 70B shapes: O and down (residual epilogue) at both, gate/up
  // only with K >= 8192 (its 8B shape was 10 % slower); QKV stays on mma.sync
  p.tc = batch > 16 && (epi == kEpiResid || (epi == kEpiSwiglu && p.n_groups >= 64));
  if (p.tc) p.nt = 4;
  // ring stage = weight unit + activation tile; as deep as lets the target
  // number of CTAs share an SM (5 up to batch 8, 3 up to 16, 2 beyond)
  // (mma.sync: rounded to 128 bytes, so every stage and its tile start on a
  // 128-byte boundary for the tensor copy)
  p.stage_bytes = p.tc ? kTcStage : (kUnitBytes + batch * kTileLd * 2 + 127) & ~127;
  const int misc = p.tc ? kTcMisc : 32 * 4 + 16 + 2 * kMaxRing * 8;
  const int per_sm = batch <= 8 ? 5 : (p.tc ? 2 : 3);
  const int budget = 232448 / per_sm - 1024 - misc - 2048 - (p.tc ? 1024 : 128);  // reserve, static arrays, alignment
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
  p.smem = (size_t)p.off_misc + misc + (p.tc ? 1024 : 128);  // the base is rounded up (1024 / 128 bytes)
  // splits: balance waves of resident CTAs; each extra split costs a partial
  // write and a share of the reduction.  The search stops at s_cap, which
  // depends only on the shape, the batch and the SM count (the CTAs that
  // shared memory admits per SM, not the runtime occupancy answer), so one
  // workspace size covers every plan: up to four waves of such CTAs over the
  // row blocks (plans of several waves let CTAs leave early, which lets the
  // next kernel start streaming its weights under programmatic launch).
  const int fit_max = std::max(1, std::min(16, 233472 / (int)(p.smem + 1024)));
  p.s_cap = std::min(p.n_groups, std::max(1, (4 * n_sm * fit_max + p.n_rb - 1) / p.n_rb));
  // QKV, O and down on the mma.sync kernels from batch 2 on: the splits of a
  // row block form one cluster and reduce in distributed shared memory, which
  // removes the global records, the arrival and the reload from each tail and
  // spreads the epilogue over the cluster (8B batch 8: 71.0 -> 61.7 µs per
  // block-step, batch 32 ragged: 145 -> 124; the QKV epilogue of 32 sequences
  // no longer runs in one CTA).  At batch 1 clusters of up to 16 CTAs are
  // placed more slowly than single CTAs while the previous kernel still holds
  // SM slots, which costs more than the shorter tail saves (8B: 52.8 vs 62.4
  // µs), and gate/up (hundreds of row blocks, a short SwiGLU tail) lost 2-6 µs
  // to whole-cluster waves: both keep the global records.  The records-only
  // QKV (kEpiQkvRec) has no epilogue here and writes global records too.
  p.cluster = !p.tc && batch > 1 && epi != kEpiSwiglu && epi != kEpiQkvRec;
  const int fit = p.tc ? resident_tc(epi, p.smem) : resident_ctas(batch == 1 ? 0 : p.nt, epi, p.smem);
  const int s_max =
      p.cluster ? std::min({p.s_cap, kMaxProjCluster, max_proj_cluster(batch == 1 ? 0 : p.nt, epi, p.smem)}) : p.s_cap;
  const long long slots = (long long)n_sm * std::min(fit > 0 ? fit : 1, fit_max);
  int best_s = 1;
  double best = 1e30;
  for (int s = 1; s <= s_max; ++s) {
    const long long items = (long long)p.n_rb * s;
    long long waves = (items + slots - 1) / slots;
    if (p.cluster) {
      // whole clusters per wave
      const int c = active_clusters(batch == 1 ? 0 : p.nt, epi, p.smem, s);
      if (c > 0) waves = std::max(waves, ((long long)p.n_rb + c - 1) / c);
    }
    const int per = (p.n_groups + s - 1) / s;
    const double cost = (double)waves * (per + 3) * (s > 1 ? 1.1 : 1.0);
    if (cost < best - 1e-9) {
      best = cost;
      best_s = s;
    }
  }
  if (force_split > 0) best_s = force_split < s_max ? force_split : s_max;
  p.S = best_s;
  p.rec_floats = batch * kRecLd;
  // split records in global memory (none with the cluster reduction); a
  // workspace reserves them for s_cap whatever the mode
  p.part_floats = p.cluster ? 0 : (size_t)p.n_rb * p.S * p.rec_floats;
  p.part_cap_floats = (size_t)p.n_rb * p.s_cap * p.rec_floats;
  return p;
}

cudaError_t launch_projection(int epi, const ProjPlan& p, ProjArgs a, cudaStream_t st, bool pdl) {
  a.S = p.S;
  a.cluster = p.cluster ? 1 : 0;
  a.part_stride = p.S;
  a.n_groups = p.n_groups;
  a.ring = p.ring;
  a.stage_bytes = p.stage_bytes;
  a.off_misc = p.off_misc;
  a.rec_floats = p.rec_floats;
  const int grid = p.n_rb * p.S;
  if (p.tc) {  // residual and SwiGLU epilogues only
    if (epi == kEpiResid) return launch_tc<kEpiResid>(a, grid, p.smem, st, pdl);
    return launch_tc<kEpiSwiglu>(a, grid, p.smem, st, pdl);
  }
  if (epi == kEpiResid) return launch_nt<kEpiResid>(p.nt, a, grid, p.smem, st, pdl);
  if (epi == kEpiSwiglu) return launch_nt<kEpiSwiglu>(p.nt, a, grid, p.smem, st, pdl);
  if (epi == kEpiQkvRec) return launch_nt<kEpiQkvRec>(p.nt, a, grid, p.smem, st, pdl);
  return launch_nt<kEpiQkv>(p.nt, a, grid, p.smem, st, pdl);
}

}  // namespace futr
