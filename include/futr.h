/*
 * futr.h -- C ABI of libfutr.so: the INT4-weight / INT4-KV decode step of a
 * Llama-style Transformer block on GB300 (sm_103a).
 *
 * The operations follow "FuTransformer: FP8 prefill and INT4 decode for
 * Llama-style inference on Hopper" (abstract) and its English explainer "FP8
 * Prefill + INT4 Decode: New Optimization for Llama Inference on Hopper"
 * (sections "FP8 Prefill: fusing GEMM and epilogue all the way" for the gain
 * folding and direct KV-cache placement, "INT4 Decode: letting dequantization
 * feed directly into MMA operands" for the INT4 projections and the INT4
 * KV-cache copy, and the paragraph on the block-diagonal Hadamard transform).
 *
 * Conventions shared by every call
 *  - Every buffer argument is a DEVICE pointer unless its name ends in _host.
 *    All device buffers are owned by the caller; the library allocates no
 *    device memory.  Buffers must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on that stream unless stated otherwise.
 *  - Host-detectable errors (bad shapes, null pointers, sizes) are returned
 *    immediately and nothing is launched.  Errors found on the device (a
 *    position outside the cache, a bad blob header, a wait that ran out) set
 *    an error word in the workspace; futr_check() returns it.  No kernel traps.
 *  - bf16 and fp16 values are passed as uint16_t bit patterns.
 *  - Supported shapes: head_dim 64 or 128; group 128; had_block a power of two
 *    between 2 and head_dim; hidden, n_q_heads*head_dim, inter multiples of
 *    128; n_q_heads a multiple of n_kv_heads with at most 16 query heads per
 *    kv-head; batch 1..32; KV capacity up to 65536 positions per sequence.
 */
#ifndef FUTR_H_
#define FUTR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t futr_status;
#define FUTR_OK                0
#define FUTR_ERR_INVALID_ARG   1  /* null pointer, size too small, index out of range */
#define FUTR_ERR_UNSUPPORTED   2  /* shape or batch outside the supported set         */
#define FUTR_ERR_CUDA          3  /* a CUDA runtime call failed                       */
#define FUTR_ERR_OUT_OF_RANGE  4  /* device: pos[b] outside [0, capacity)             */
#define FUTR_ERR_TIMEOUT       5  /* device: a bounded wait ran out                   */
#define FUTR_ERR_BAD_BLOB      6  /* device or host: weight blob header mismatch      */
#define FUTR_ERR_NOT_PD        7  /* GPTQ: a dampened Hessian is not positive definite */
#define FUTR_ERR_CORRUPT       8  /* device: guard words after a region overwritten    */
#define FUTR_ERR_BOUNDS        9  /* device, debug build: an index failed its check    */

/* Shape of one decoder block. */
typedef struct futr_shape {
  int32_t hidden;      /* model width H                                  */
  int32_t n_q_heads;   /* query heads Hq                                 */
  int32_t n_kv_heads;  /* key/value heads Hkv (grouped-query attention)  */
  int32_t head_dim;    /* d                                              */
  int32_t inter;       /* SwiGLU intermediate width I                    */
  int32_t group;       /* INT4 scale group along the input dim (128)     */
  int32_t had_block;   /* Hadamard block size along head_dim             */
  float rms_eps;       /* RMSNorm epsilon (1e-5)                         */
  float rope_theta;    /* RoPE base (500000)                             */
} futr_shape;

/* INT4 KV cache descriptor: plain data filled by futr_kv_init, kept by the
 * caller (host memory).  `base` is the caller's device buffer. */
typedef struct futr_kv {
  futr_shape shape;
  int32_t n_layers, max_batch, capacity;   /* capacity: positions per sequence */
  int32_t _pad;
  void* base;
  uint64_t bytes;
  uint64_t stream_bytes;                   /* bytes of one (layer, seq, kv-head) stream */
  uint64_t rope_offset;                    /* cos/sin table [capacity][d/2] float2      */
  uint64_t err_offset;                     /* int32 error word of futr_kv_append        */
  uint64_t magic;
} futr_kv;

/* Workspace descriptor: plain data filled by futr_workspace_init.  The
 * offsets name the intermediate activations of the last decode call. */
typedef struct futr_ws {
  futr_shape shape;
  int32_t max_batch, capacity, n_sm, _pad;
  void* base;
  uint64_t bytes;
  uint64_t off_err;      /* int32 error word                                   */
  uint64_t off_qrot;     /* fp32 [b][Hq][d]   rotated query                     */
  uint64_t off_o;        /* bf16 [b][Hq*d]    attention output (unrotated)      */
  uint64_t off_h;        /* bf16 [b][H]       residual after attention          */
  uint64_t off_a;        /* bf16 [b][I]       SwiGLU activation                 */
  uint64_t off_xin;      /* bf16 [b][H]       staging for futr_decode_block_host */
  uint64_t off_yout;     /* bf16 [b][H]                                          */
  uint64_t off_pos;      /* int32 [b]                                            */
  uint64_t off_part;     /* fp32 split-K partial sums                            */
  uint64_t part_bytes;
  uint64_t off_apart;    /* fp32 attention range records (whole-block kernel)    */
  uint64_t apart_bytes;
  uint64_t off_cnt;      /* uint32 arrival counters (self-resetting)             */
  uint64_t cnt_words;
  uint64_t magic;
} futr_ws;

/* Which projection a canonical (unpacked) view refers to. */
#define FUTR_PROJ_QKV   0   /* rows: Wq; Wk; Wv  [Hq*d + 2*Hkv*d, H], gain g_attn */
#define FUTR_PROJ_O     1   /* [H, Hq*d], no gain                                   */
#define FUTR_PROJ_GATE  2   /* [I, H], gain g_mlp                                   */
#define FUTR_PROJ_UP    3   /* [I, H], gain g_mlp                                   */
#define FUTR_PROJ_DOWN  4   /* [H, I], no gain                                      */

/* Human-readable text for a status code (static string). */
const char* futr_status_string(futr_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t futr_version(void);

/* Bytes of the packed weight blob of one block for `shape`. */
futr_status futr_weights_size(const futr_shape* shape, size_t* bytes);

/*
 * Offline packer.  The abstract folds the fixed RMSNorm gain into the weights
 * and quantizes the projection weights to INT4 by rounding to nearest; the
 * explainer's INT4 Decode section stores them in the tensor cores' fragment
 * layout.
 *
 * Inputs are fp32 device matrices in nn.Linear layout [out, in], row-major:
 * wq [Hq*d, H], wk/wv [Hkv*d, H], wo [H, Hq*d], wgate/wup [I, H], wdown [H, I],
 * and the RMSNorm gains g_attn, g_mlp [H].  For every projection W' = W diag(g)
 * (g_attn for q/k/v, g_mlp for gate/up, none for o/down) is rounded once to
 * fp32, then each (output row, 128-input group) gets the fp16 scale
 * s = fp16(max|W'| / 7) (fp32 division, nearest-even; saturates at 65504) and
 * codes c = clamp(round_half_even(fp32(W' / s)), -8, 7) (all 0 when s == 0).
 * The blob (`blob_bytes` >= futr_weights_size) receives a 256-byte header and
 * four sections (QKV, O, gate/up interleaved per 64 rows, down) of 8448-byte
 * units: 128 output rows x 128 inputs of nibbles in mma.m16n8k16 A-fragment
 * order, then the units' 128 fp16 scales.
 */
futr_status futr_pack_weights(const futr_shape* shape,
                              const float* wq, const float* wk, const float* wv,
                              const float* wo, const float* wgate, const float* wup,
                              const float* wdown, const float* g_attn, const float* g_mlp,
                              void* blob, size_t blob_bytes, void* stream);

/* Bytes of device scratch futr_pack_weights_gptq needs for `shape`: two
 * float64 K x K matrices for the largest input width K of the block (the
 * intermediate size), a float64 copy of the largest projection, and its codes. */
futr_status futr_gptq_scratch_size(const futr_shape* shape, size_t* bytes);

/*
 * GPTQ packer: the same blob as futr_pack_weights (same header, layout, scale
 * rule s = fp16(max|w| / 7) and code range), with the codes chosen by GPTQ.
 * The abstract quantizes the decode weights with GPTQ in the round-to-nearest
 * INT4 format; the explainer's accuracy section describes it as using
 * calibration data and approximate second-order information.  The steps are
 * those of the published GPTQ algorithm (Frantar et al., 2022), columns in
 * natural order, no activation reordering:
 *   H' = H with every dead input (H_jj = 0) set to H_jj = 1 and its weight
 *        column to 0, then H' += damp * mean(diag H') * I;
 *   U  = upper Cholesky factor of H'^-1 (H'^-1 = U^T U);
 *   for j = 0..K-1 on a float64 copy of W' = fp32(W diag(g)): at the first
 *   input of each 128-group the group's scales are taken from its current
 *   weights (rounded to fp32); c_j = clamp(rint(fp32(w_j) / s), -8, 7);
 *   e = (w_j - c_j s) / U_jj; W[:, j+1:] -= e U[j, j+1:].
 * Everything runs in float64 on the device (blocked Cholesky and triangular
 * inverse, the sweep in 128-column blocks with the trailing update as a GEMM);
 * the float64 additions come in another order than the column-by-column sweep.
 *
 * Hessians (float64 device, symmetric, [K, K] for the projection's input
 * width K): h_attn [H, H] of the normalized block input (QKV), h_o
 * [Hq*d, Hq*d] of the attention output (O), h_mlp [H, H] of the normalized
 * residual (gate and up), h_down [I, I] of the SwiGLU output (down); a
 * calibration set X [n, K] gives H = (2/n) X^T X.  damp > 0 (0.01 is usual).
 * scratch: futr_gptq_scratch_size bytes, 256-byte aligned; its contents are
 * undefined afterwards.  Other arguments as for futr_pack_weights.
 * Synchronous: returns after `stream` has finished.  FUTR_ERR_NOT_PD when a
 * dampened Hessian has a non-positive Cholesky pivot (the blob is then not
 * usable).
 */
futr_status futr_pack_weights_gptq(const futr_shape* shape,
                                   const float* wq, const float* wk, const float* wv,
                                   const float* wo, const float* wgate, const float* wup,
                                   const float* wdown, const float* g_attn, const float* g_mlp,
                                   const double* h_attn, const double* h_o, const double* h_mlp,
                                   const double* h_down, double damp,
                                   void* scratch, size_t scratch_bytes,
                                   void* blob, size_t blob_bytes, void* stream);

/*
 * Canonical view of one packed projection (for verification): codes int8
 * [rows, cols] row-major in [-8, 7] and fp16 scales [rows, cols/128], with
 * rows/cols as listed for FUTR_PROJ_*.  Device outputs.
 */
futr_status futr_unpack_weights(const futr_shape* shape, const void* blob, int32_t which,
                                int8_t* codes, uint16_t* scales, void* stream);

/* Bytes of an INT4 KV cache for n_layers x max_batch sequences of `capacity`
 * positions (capacity is rounded up to a multiple of 16). */
futr_status futr_kv_size(const futr_shape* shape, int32_t n_layers, int32_t max_batch,
                         int32_t capacity, size_t* bytes);

/* Zero `kv_mem`, write the RoPE cos/sin table (float64 evaluation rounded to
 * fp32) and the guard words after each region (see futr_check), and fill the
 * host descriptor `kv`.  Asynchronous on `stream`. */
futr_status futr_kv_init(const futr_shape* shape, int32_t n_layers, int32_t max_batch,
                         int32_t capacity, void* kv_mem, size_t kv_bytes, futr_kv* kv,
                         void* stream);

/*
 * INT4 KV-cache copy writer.  The abstract keeps an INT4 copy of the KV cache
 * and rotates it block-diagonally with a Hadamard matrix, which lowers the
 * quantization error that outlier channels cause.  For sequences seq0 .. seq0+batch-1 of layer `layer`,
 * append n_tok tokens at positions pos[b] .. pos[b]+n_tok-1 (pos: device int32
 * [batch]).  k, v: bf16 [batch][Hkv][n_tok][d] (already position-encoded).
 * Each (token, kv-head) vector is widened to fp32, rotated by the fp32 fast
 * Walsh-Hadamard transform in blocks of had_block (stage s pairs i and i+2^s,
 * ascending s, then one multiply by fp32(1/sqrt(had_block))) and quantized to
 * INT4 with one fp16 scale, by the same rule as the weights.  Keys are stored
 * in mma B-fragment order per 8 positions, values per 16 positions.
 * Positions outside [0, capacity) set FUTR_ERR_OUT_OF_RANGE in the cache's
 * error word (see futr_check) and are skipped.
 */
futr_status futr_kv_append(const futr_kv* kv, int32_t layer, int32_t seq0, int32_t batch,
                           const int32_t* pos, int32_t n_tok, const uint16_t* k,
                           const uint16_t* v, void* stream);

/* Canonical view of cached entries 0..n_pos-1 of one sequence: codes int8
 * [Hkv][n_pos][d], fp16 scales [Hkv][n_pos], for keys and values.  Device
 * outputs. */
futr_status futr_kv_read(const futr_kv* kv, int32_t layer, int32_t seq, int32_t n_pos,
                         int8_t* k_codes, uint16_t* k_scales, int8_t* v_codes,
                         uint16_t* v_scales, void* stream);

/* Bytes of the workspace for decode calls with batch <= max_batch over caches
 * of `capacity` positions. */
futr_status futr_workspace_size(const futr_shape* shape, int32_t max_batch, int32_t capacity,
                                size_t* bytes);

/* Zero the workspace (its counters must start at 0), write the guard words
 * after each region (see futr_check) and fill `ws`.  The current CUDA device
 * must be the one the workspace lives on. */
futr_status futr_workspace_init(const futr_shape* shape, int32_t max_batch, int32_t capacity,
                                void* ws_mem, size_t ws_bytes, futr_ws* ws, void* stream);

/*
 * One decode step of one block for `batch` sequences (abstract: decode runs on
 * INT4 projection weights and the INT4 copy of the KV cache):
 *   r1 = 1/sqrt(mean(x^2)+eps);  [q;k;v] = r1 * (W'qkv x);  RoPE(q, k) at pos[b];
 *   q' = H q / sqrt(n) (fp32); the new k, v are rotated, quantized and stored in
 *   slot pos[b] of the cache (direct KV-cache placement);
 *   o = bf16(H^T softmax(q' K'^T / sqrt(d)) V' / sqrt(n)) over slots 0..pos[b]
 *   (grouped-query: q-head h reads kv-head h / (Hq/Hkv));
 *   h = bf16(x + Wo o);  r2 = 1/sqrt(mean(h^2)+eps);
 *   a = bf16(silu(r2 W'gate h) * (r2 W'up h));  y = bf16(h + Wdown a).
 * x, y: bf16 [batch][H] (may not alias).  pos: device int32 [batch], the number
 * of tokens already cached per sequence (sequence b uses cache slot b).
 * blob: packed weights of this layer.  Five kernels launched back to back with
 * programmatic dependent launch.  When a kv-head has at most 8 query heads
 * the QKV kernel leaves its split-K partial sums in the workspace
 * and the attention kernel adds them and runs the head epilogue (RMSNorm
 * factor, RoPE, rotation, the new token's quantization and placement);
 * FUTR_QKV_DEFER=0 keeps that epilogue in the QKV kernel.  Either way the
 * workspace's qrot holds q' afterwards.  With the environment variable
 * FUTR_PERSISTENT=1 and batch 1..16, one persistent kernel runs the whole step
 * instead (launched in plain stream order with all CTAs resident; it assumes no
 * other kernel holds the GPU's SMs meanwhile, else a bounded wait may report
 * FUTR_ERR_TIMEOUT).  Capturable in a CUDA graph.
 */
futr_status futr_decode_block(const uint16_t* x, const void* blob, const futr_kv* kv,
                              int32_t layer, int32_t batch, const int32_t* pos, uint16_t* y,
                              const futr_ws* ws, void* stream);

/* As futr_decode_block run as five kernels at every batch, with a CUDA event
 * recorded before each kernel and after the last (without programmatic
 * overlap).  Synchronizes
 * `stream` and writes the five kernel times in milliseconds to
 * stage_ms_host[5] (QKV, attention, O, gate/up, down; the QKV head epilogue
 * counts in the attention time when it runs there, see futr_decode_block). */
futr_status futr_decode_block_timed(const uint16_t* x, const void* blob, const futr_kv* kv,
                                    int32_t layer, int32_t batch, const int32_t* pos,
                                    uint16_t* y, const futr_ws* ws, void* stream,
                                    float* stage_ms_host);

/* As futr_decode_block with HOST input and output: copies x_host (bf16
 * [batch][H]) into the workspace, runs the block on pos_host (int32 [batch])
 * and writes y_host, and synchronizes `stream`.  When pos_host and y_host are
 * both page-locked and mapped for the device (cudaHostAlloc / cudaHostRegister
 * memory on a unified-address system), the kernels read pos and write y there
 * directly; otherwise they are copied through the workspace's staging rows.
 * y_host must not be read before the call returns. */
futr_status futr_decode_block_host(const uint16_t* x_host, const void* blob, const futr_kv* kv,
                                   int32_t layer, int32_t batch, const int32_t* pos_host,
                                   uint16_t* y_host, const futr_ws* ws, void* stream);

/*
 * futr_decode_block without a caller workspace, for callers that cannot
 * allocate device memory (a plugin inside a runtime that owns every
 * allocation, code under a fixed allocator or memory budget, or a program
 * that must not call cudaMalloc at run time).  The paper has no counterpart:
 * this is a deployment variant of the same step.  Arguments as for
 * futr_decode_block; x, blob, kv, pos and y are still the caller's.
 *
 * All scratch memory (intermediate activations, partial sums, counters) is a
 * 48 MiB array inside the library that every device loading the library keeps
 * until exit.  The call allocates nothing and calls no allocating routine.
 * - Returns FUTR_ERR_UNSUPPORTED, launching nothing, when this shape and batch
 *   need more than 48 MiB of scratch (the size does not depend on the cache's
 *   capacity; the 8B- and 70B-shaped blocks need about 38 MB at batch 32 on a
 *   152-SM GPU, less at smaller batches).
 * - The first call on a device resolves the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.
 * - Every call uses the same array and clears its counters first, so calls
 *   whose work overlaps on the GPU (other streams, other threads) race;
 *   serialize them.
 * - Device-detected errors land in the array's error word, which the next
 *   call clears; use futr_decode_block and futr_check when they must be read.
 */
futr_status futr_decode_block_noalloc(const uint16_t* x, const void* blob, const futr_kv* kv,
                                      int32_t layer, int32_t batch, const int32_t* pos, uint16_t* y,
                                      void* stream);

/*
 * One complete decode step of an n_layers-block model: the abstract of
 * "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
 * Hopper" times a complete Llama-3.1-8B decode step (the blocks plus the
 * embedding, the final norm and the LM head).
 *   x = embedding[tokens[b]];  for l < n_layers: x = futr_decode_block(x, blobs[l],
 *   layer l);  r = 1/sqrt(mean(x^2)+eps);  xg = bf16(fp32(g_final * x));
 *   logits[b][v] = r * sum_k lm_head[v][k] * xg[k]   (fp32 accumulation).
 * No INT4 projection follows the final norm, so its gain cannot be folded into
 * INT4 codes: the LM head stays bf16 and the gain scales the activation.
 * tokens: device int32 [batch]; a token outside [0, vocab) sets
 * FUTR_ERR_OUT_OF_RANGE and reads as a zero embedding.  embedding, lm_head:
 * device bf16 [vocab][H], 16-byte aligned, vocab a multiple of 64.  blobs: HOST
 * array of n_layers device pointers (packed weights of layers 0..n_layers-1;
 * kv must hold at least n_layers layers).  pos as for futr_decode_block.
 * g_final: device fp32 [H].  logits: device fp32 [batch][vocab].  The residual
 * stream passes through the workspace's staging rows, which the step uses in
 * place of futr_decode_block_host's.  Launches embedding, 5 kernels per block,
 * final norm and LM head with programmatic dependent launch; capturable.
 */
futr_status futr_decode_step(const int32_t* tokens, const uint16_t* embedding, int32_t vocab,
                             const void* const* blobs, int32_t n_layers, const futr_kv* kv,
                             int32_t batch, const int32_t* pos, const float* g_final,
                             const uint16_t* lm_head, float* logits, const futr_ws* ws,
                             void* stream);

/* Compare the guard words of `ws` and `kv` with their pattern (every region of
 * a workspace and of a cache is followed by 256 guard bytes that
 * futr_workspace_init / futr_kv_init fill and no kernel writes; an overwritten
 * guard sets FUTR_ERR_CORRUPT, and stays overwritten until the buffer is
 * initialised again), synchronize `stream`, then return (and clear) the first
 * nonzero device error word of the workspace `ws` and of the cache `kv` (either
 * may be NULL), or FUTR_ERR_CUDA if a CUDA error is pending. */
futr_status futr_check(const futr_ws* ws, const futr_kv* kv, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FUTR_H_ */
