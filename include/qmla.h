/*
 * qmla.h - C ABI of the low-bit Multi-Head Latent Attention (MLA) decode library.
 *
 * What the method computes (QuantMLA, as described by the pages
 * "QuantMLA: INT4 (and INT2) for both halves of the MLA cache", TL;DR and the
 * mermaid flowchart, and "Hugging Face Releases QuantMLA", section
 * "Engineering Trade-offs and Performance"):
 *   - every cached token keeps two things: a content latent (the shared K/V
 *     source, d_c = 512 channels) and a small decoupled RoPE key (the position
 *     part, d_r = 64 channels);
 *   - the content latent is stored at INT4 or INT2, the RoPE key at INT4
 *     ("C4R4" / "C2R4"), and the RoPE path is never taken below INT4;
 *   - for the comparison with generic quantizers, which give both halves one
 *     bit width ("Key findings" of the first page), the RoPE key can also be
 *     stored at INT2 ("C4R2" / "C2R2"); these two formats are served by the
 *     CUDA-core decode kernel only;
 *   - a native low-bit attention kernel unpacks and dequantizes inside the
 *     attention computation; nothing is expanded back to a 16-bit cache.
 * The learned path-specific transforms are folded into the model weights
 * offline (flowchart; "Key findings", function-aligned objectives), so the
 * queries and latents handed to this library are already transformed.
 *
 * Parameters the pages leave open and this library fixes:
 *   group size 64 channels; asymmetric quantization with one fp16 scale and one
 *   fp16 zero per (token, 64-channel group); a paged cache of 64-token blocks;
 *   absorbed-query decode with softmax scale 1/sqrt(192) supplied by the caller.
 *
 * ---------------------------------------------------------------------------
 * Quantizer (per token, per group of 64 channels, b = 4 or 2 bits,
 * levels = 2^b - 1):
 *   mn, mx  = min and max of the group (exact)
 *   grid    = the smallest power of two u = 2^E, -24 <= E <= 5, for which the
 *             integers Z = floor(mn / u) and
 *             M = max(1, ceil((mx - Z*u) / (levels*u)))   (quotient rounded up)
 *             satisfy |Z| <= 2047 and |Z + levels*M| <= 2047; the search starts
 *             at E = max(-24, ilogb(mx - mn) - 12) (difference rounded down),
 *             a lower bound; every step is exact (no rounding decides E, Z
 *             or M)
 *   z       = Z*u, s = M*u, both stored as binary16 (exactly)
 *   code_i  = clamp(rint((x_i - z) / s), 0, levels), the subtraction and the
 *             division in binary32 rounded to nearest-even, rint half to even
 * Then z <= mn and z + levels*s >= mx, so every element is reproduced within
 * s/2 (plus binary32 rounding) by x_hat = code*s + z, and every x_hat
 * (= (Z + code*M)*u, an integer of at most 11 bits times a power of two) is
 * exactly a binary16 number: the tensor cores multiply exactly the value the
 * quantizer defines.  For groups containing zero the step s exceeds the ideal
 * (mx - mn)/levels by at most 16/1023 (INT4) or 4/1023 (INT2) relative.
 *
 * Code packing inside each little-endian 32-bit word (8 INT4 or 16 INT2 codes
 * of consecutive channels c0 .. c0+7 / c0+15): the low 16 bits hold the even
 * channels c0, c0+2, ... in increasing order, the high 16 bits the odd
 * channels c0+1, c0+3, ....  INT4: bits [4k, 4k+4) = channel c0 + 2k for k < 4,
 * channel c0 + 2(k-4) + 1 for k >= 4.  INT2: bits [2k, 2k+2) = channel c0 + 2k
 * for k < 8, channel c0 + 2(k-8) + 1 for k >= 8.
 *
 * Block layout (one block = 64 token slots; slot = position % 64).  A block is
 * split into two "halves": half h holds content channels 256h .. 256h+255
 * (content groups 4h .. 4h+3) and RoPE channels 32h .. 32h+31.
 *   C4R4 (CB = 32 code bytes per content group per token, RB = 16, HALF = 10240 B)
 *   C2R4 (CB = 16,                                        RB = 16, HALF =  6144 B)
 *   C4R2 (CB = 32,                                        RB =  8, HALF =  9728 B)
 *   C2R2 (CB = 16,                                        RB =  8, HALF =  5632 B)
 *     half h at byte h*HALF:
 *       content codes   [4 groups][64 slots][CB]             (4*64*CB B)
 *       RoPE codes      [64 slots][RB] (32 channels, INT4 or INT2) (64*RB B)
 *       content s/z     [4 groups][64 slots][2] binary16 (scale, zero) (1024 B)
 *     RoPE s/z at byte 2*HALF: [64 slots][2] binary16 (scale, zero) (256 B);
 *     the RoPE key is one 64-channel group, so both halves share it.
 *     Block bytes: C4R4 20736 (324 B/token), C2R4 12544 (196 B/token),
 *     C4R2 19712 (308 B/token), C2R2 11520 (180 B/token).
 *   BF16 (comparison cache, no quantization, HALF = 36864 B)
 *     half h at byte h*HALF:
 *       content  [4 groups][64 slots][64] bfloat16   (32768 B)
 *       RoPE     [64 slots][32] bfloat16             (4096 B)
 *     Block bytes: 73728 (1152 B/token).
 * Every region starts on a 256-byte boundary inside the block; block i of
 * the pool starts at blocks + i * qmla_block_bytes(format), so the pool base
 * must be 256-byte aligned.
 *
 * ---------------------------------------------------------------------------
 * Decode (per sequence b and head h, L = seq_lens[b] tokens):
 *   s_t = (q_c[h] . c_hat_t + q_r[h] . k_hat_t) * softmax_scale
 *   LSE = ln sum_t exp(s_t)                      (natural log, scale included)
 *   O   = sum_t exp(s_t - LSE) * c_hat_t         (content latent only, 512)
 * L = 0 gives O = 0 and LSE = -inf.
 *
 * Conventions for every call below:
 *   - all array pointers are caller-owned DEVICE memory unless stated;
 *     the library never allocates, frees or retains them;
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream); work is enqueued asynchronously and the call returns at once;
 *   - the return value is QMLA_OK or a negative QMLA_ERR_* code; a non-OK
 *     return means nothing was enqueued;
 *   - faults the host cannot see (a block id outside the pool, a sequence
 *     longer than its block table or than max_seq_len, a bounded device wait
 *     that gave up) are OR-ed as QMLA_STATUS_* bits into *status_dev, a
 *     caller-owned device int32 that the caller zeroes; the kernels skip the
 *     offending work instead of faulting.  qmla_read_status() fetches it.
 */
#ifndef QMLA_H_
#define QMLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMLA_D_C 512          /* content latent channels */
#define QMLA_D_R 64           /* decoupled RoPE key channels */
#define QMLA_GROUP 64         /* channels per quantization group */
#define QMLA_BLOCK_TOKENS 64  /* token slots per cache block */

typedef enum {
  QMLA_C4R4 = 0, /* content INT4, RoPE INT4 */
  QMLA_C2R4 = 1, /* content INT2, RoPE INT4 */
  QMLA_BF16 = 2, /* unquantized bfloat16 comparison cache */
  QMLA_C4R2 = 3, /* content INT4, RoPE INT2 (equal-bits comparison) */
  QMLA_C2R2 = 4  /* content INT2, RoPE INT2 (equal-bits comparison) */
} qmla_format;

enum {
  QMLA_OK = 0,
  QMLA_ERR_INVALID_ARG = -1, /* null pointer, negative size, misaligned pointer */
  QMLA_ERR_UNSUPPORTED = -2, /* format or head count this build does not serve */
  QMLA_ERR_CAPACITY = -3,    /* request larger than a fixed limit of the call */
  QMLA_ERR_WORKSPACE = -4,   /* workspace smaller than qmla_decode_workspace_bytes */
  QMLA_ERR_CUDA = -5,        /* a CUDA runtime call or kernel launch failed */
  QMLA_ERR_DEVICE = -6       /* qmla_read_status found a device status bit set */
};

/* Device status bits OR-ed into *status_dev. */
#define QMLA_STATUS_BAD_BLOCK 0x1 /* block id < 0 or >= num_blocks; block skipped */
#define QMLA_STATUS_BAD_LEN 0x2   /* position/length outside the block table or max_seq_len */
#define QMLA_STATUS_TIMEOUT 0x4   /* a bounded device wait gave up; output invalid */
#define QMLA_STATUS_BAD_QUERY 0x8 /* a query value overflows binary16 (|q| > 65504) in a
                                     tensor-core decode; rows holding it are not valid */

/* Bytes of one 64-token block in `format` (20736 / 12544 / 73728 / 19712 /
 * 11520), 0 for an unknown format.  Layout in the comment at the top of this file. */
size_t qmla_block_bytes(int format);

/* qmla_append - quantize and pack new tokens into the paged cache.
 * Operation: the two quantizers of the flowchart of "QuantMLA: INT4 (and INT2)
 * for both halves of the MLA cache" (content quant INT4 or INT2, RoPE quant
 * INT4), with the rounding rules at the top of this file.
 *   blocks            [num_blocks * qmla_block_bytes(format)] bytes, written
 *   block_table       [batch][max_blocks_per_seq] int32 block ids
 *   positions         [batch] int32: slot index of the first new token of each
 *                     sequence (its current length); the caller advances it
 *   latent            [batch][n_new][512] bfloat16, row-major
 *   rope_k            [batch][n_new][64]  bfloat16 (RoPE already applied)
 *   status_dev        device int32, status bits OR-ed in
 * Token i of sequence b goes to slot (positions[b]+i) % 64 of block
 * block_table[b][(positions[b]+i) / 64].  Bit-exact and independent of how
 * the tokens are batched.  Inputs must be finite with |x| < 32768 (so that
 * scale and zero fit binary16).  Errors: INVALID_ARG (null pointer, batch,
 * n_new or max_blocks_per_seq < 0, num_blocks < 1), UNSUPPORTED (format),
 * CUDA (launch).  A slot beyond the block table or a block id outside the
 * pool sets a status bit and that token is skipped. */
int qmla_append(int format, void* blocks, int64_t num_blocks,
                const int32_t* block_table, int32_t max_blocks_per_seq,
                const int32_t* positions, int32_t batch, int32_t n_new,
                const void* latent, const void* rope_k,
                int32_t* status_dev, void* stream);

/* qmla_append_advance - qmla_append, then positions[b] += n_new for every
 * sequence, on the device and in the same call (positions is written).  For
 * a decode step (n_new = 1) this is one kernel: each sequence's CTA advances
 * its own position once it has read it.  Errors as qmla_append; a token
 * that is skipped for a bad slot or block id still advances its position. */
int qmla_append_advance(int format, void* blocks, int64_t num_blocks,
                        const int32_t* block_table, int32_t max_blocks_per_seq,
                        int32_t* positions, int32_t batch, int32_t n_new,
                        const void* latent, const void* rope_k,
                        int32_t* status_dev, void* stream);

/* Workspace bytes qmla_decode needs for these sizes (split partials and the
 * per-sequence merge table); 0 for unsupported arguments. */
size_t qmla_decode_workspace_bytes(int format, int32_t batch, int32_t heads,
                                   int32_t max_seq_len);

/* qmla_decode - absorbed-query MLA decode over the low-bit paged cache.
 * Operation: the "native low-bit MLA attention kernel" that "unpacks and
 * dequantizes inside attention" ("QuantMLA: INT4 (and INT2) for both halves
 * of the MLA cache", section "Key findings"; flowchart node "Low-bit kernel"),
 * computing the decode formula at the top of this file with the context split
 * across CTAs and merged by log-sum-exp.
 *   blocks, block_table, max_blocks_per_seq   as for qmla_append (read only)
 *   seq_lens          [batch] int32 device: tokens cached per sequence
 *   max_seq_len       host bound on seq_lens used to size the split plan
 *   heads             query heads; 16 and 128 use the tensor-core kernels,
 *                     any multiple of 16 up to 256 is served
 *   q_c               [batch][heads][512] bfloat16 absorbed content queries
 *   q_r               [batch][heads][64]  bfloat16 RoPE queries
 *   softmax_scale     e.g. 1/sqrt(192)
 *   out               [batch][heads][512] bfloat16, written
 *   lse               [batch][heads] float32 natural-log LSE, written
 *   workspace         device scratch of >= qmla_decode_workspace_bytes(...)
 *                     bytes, 256-byte aligned; contents need no initialization
 * The tensor-core kernels take queries as binary16 operands: |q| must stay
 * below 65504; with the BF16 cache they convert cache values to binary16 as
 * well, so those must stay below 65504 too (values under 2^-14 keep only
 * binary16's subnormal precision).  Errors: INVALID_ARG, UNSUPPORTED (format, heads), WORKSPACE,
 * CUDA.  Sequences longer than max_seq_len or their block table set
 * QMLA_STATUS_BAD_LEN and are truncated. */
int qmla_decode(int format, const void* blocks, int64_t num_blocks,
                const int32_t* block_table, int32_t max_blocks_per_seq,
                const int32_t* seq_lens, int32_t max_seq_len,
                int32_t batch, int32_t heads,
                const void* q_c, const void* q_r, float softmax_scale,
                void* out, float* lse,
                void* workspace, size_t workspace_bytes,
                int32_t* status_dev, void* stream);

/* qmla_decode_multi - decode of q_len query tokens per sequence (a
 * multi-token prediction or speculative-verification step), the last q_len
 * tokens of each cached sequence: query i sits at position L - q_len + i and
 * attends causally, to cached tokens 0 .. L - q_len + i (none when that is
 * negative: O = 0, LSE = -inf).  The pages describe single-token decode only;
 * this is the same attention over the same cache with a causal mask.
 *   q_c   [batch][q_len][heads][512], q_r [batch][q_len][heads][64] bfloat16
 *   out   [batch][q_len][heads][512] bfloat16, lse [batch][q_len][heads]
 *   workspace  >= qmla_decode_workspace_bytes(format, batch, heads * q_len, ...)
 * The kernels see heads * q_len query rows: 128 run on the tensor cores,
 * other multiples of 16 up to 256 (16 included) on the CUDA cores.  Errors: as
 * qmla_decode; INVALID_ARG for q_len < 1 or heads < 1; UNSUPPORTED when
 * heads * q_len is not served. */
int qmla_decode_multi(int format, const void* blocks, int64_t num_blocks,
                      const int32_t* block_table, int32_t max_blocks_per_seq,
                      const int32_t* seq_lens, int32_t max_seq_len,
                      int32_t batch, int32_t heads, int32_t q_len,
                      const void* q_c, const void* q_r, float softmax_scale,
                      void* out, float* lse,
                      void* workspace, size_t workspace_bytes,
                      int32_t* status_dev, void* stream);

/* Size of the library's own decode scratch used by qmla_decode_noalloc. */
#define QMLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB per device */

/* qmla_decode_noalloc - qmla_decode for callers that cannot allocate.
 * The paper has no counterpart to this call; it is a service of this library.
 * Some callers cannot allocate device memory where they decode: a serving
 * loop that must not call cudaMalloc once running (it synchronizes the whole
 * device and can fail under memory pressure), or a plugin whose host only
 * hands it a stream to enqueue work on.  This call takes the same arguments
 * as qmla_decode minus the workspace: the split partials and the merge table
 * go to a fixed QMLA_NOALLOC_SCRATCH_BYTES array in the library's device
 * memory, which every GPU that loads the library holds until process exit.
 * Nothing is allocated or freed, by the library or by any other runtime.
 *   - The first call on a device looks up that array's device address with
 *     cudaGetSymbolAddress (device current) and keeps it; make that first
 *     call before capturing the stream into a CUDA graph.
 *   - All calls share the one array, which keeps the last call's contents
 *     (no part of it needs to start at zero).  Calls whose executions
 *     overlap on the GPU (on different streams, or concurrently from several
 *     host threads) race on it: serialize them.
 *   - When the partials of the usual split do not fit, the context is split
 *     over the largest number of workers whose partials do fit; a batch
 *     whose merge table plus one partial per sequence exceeds the array
 *     (roughly batch * heads > 16000 at 512 channels) returns
 *     QMLA_ERR_CAPACITY and enqueues nothing.
 * Formats, head counts, other errors and device status bits as for
 * qmla_decode. */
int qmla_decode_noalloc(int format, const void* blocks, int64_t num_blocks,
                        const int32_t* block_table, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens, int32_t max_seq_len,
                        int32_t batch, int32_t heads,
                        const void* q_c, const void* q_r, float softmax_scale,
                        void* out, float* lse, int32_t* status_dev, void* stream);

/* qmla_decode_timeout_test - TEST HOOK for the failure path of the bounded
 * device waits; not for production use.  Same arguments as qmla_decode, for
 * 16 or 128 heads and the C4R4 / C2R4 formats only (else
 * QMLA_ERR_UNSUPPORTED).  The tensor-core kernel's dequantization warps
 * withhold a barrier arrival on the first tile (16 heads: of every worker;
 * 128 heads: of the first CTA of every CTA pair, so the second CTA's waits
 * on its partner run out too), so the waits behind it run out after their
 * 1 s limit: every role of the kernel then unwinds, the kernel exits
 * normally, QMLA_STATUS_TIMEOUT is OR-ed into *status_dev and out / lse hold
 * no valid result.  The CUDA context stays usable.  Nothing faults, traps or
 * hangs. */
int qmla_decode_timeout_test(int format, const void* blocks, int64_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t max_seq_len, int32_t batch,
                             int32_t heads, const void* q_c, const void* q_r,
                             float softmax_scale, void* out, float* lse, void* workspace,
                             size_t workspace_bytes, int32_t* status_dev, void* stream);

/* qmla_decode_step_layout - byte offsets of the packed host buffers of
 * qmla_decode_step.  Regions follow one another, each starting at the first
 * multiple of 256 bytes at or after the end of the one before (the first at
 * 0):
 *   input   latent [batch][n_new][512] bf16, rope_k [batch][n_new][64] bf16,
 *           q_c [batch][heads][512] bf16, q_r [batch][heads][64] bf16
 *           (n_new = 0: only q_c and q_r; their offsets are then 0 and
 *           after q_c, and the latent and rope_k entries are 0)
 *   output  out [batch][heads][512] bf16, lse [batch][heads] float32
 * offsets[0..7] = latent, rope_k, q_c, q_r, input bytes (the end of q_r),
 * out, lse, output bytes (the end of lse).  Returns QMLA_OK, or INVALID_ARG
 * for a null `offsets` or negative sizes.  Host-only arithmetic. */
int qmla_decode_step_layout(int32_t batch, int32_t heads, int32_t n_new, size_t* offsets);

/* Device workspace bytes qmla_decode_step needs: staging of one step's
 * input and output buffers plus qmla_decode's workspace; 0 for unsupported
 * arguments. */
size_t qmla_decode_step_workspace_bytes(int format, int32_t batch, int32_t heads,
                                        int32_t n_new, int32_t max_seq_len);

/* qmla_decode_step - one decode step of a serving loop, from host memory to
 * host memory, in one call: the step's input buffer (n_new new tokens per
 * sequence, n_new >= 0, and the queries; layout of qmla_decode_step_layout)
 * is copied to the device, the tokens are appended and every length advanced
 * by n_new (qmla_append_advance), the decode runs over the advanced lengths
 * (qmla_decode), out and lse are copied into the output buffer, and the call
 * returns once they are there (it synchronizes `stream`).  The pages' decode
 * step (append the new token's compressed latent, attend over the cache);
 * the packing of host buffers is this library's.
 *   h_in          host, >= offsets[4] bytes, read
 *   h_out         host, >= offsets[7] bytes, written
 *   seq_lens      [batch] int32 device: lengths before the step, advanced
 *   max_seq_len   bound on the advanced lengths
 *   workspace     device, >= qmla_decode_step_workspace_bytes(...) bytes,
 *                 256-byte aligned; contents need no initialization
 * Other arguments as for qmla_append_advance and qmla_decode.  Page-locked
 * host buffers (cudaHostAlloc) let the copies run asynchronously at full
 * speed; pageable ones work too.  Errors: those of qmla_append_advance and
 * qmla_decode, checked before anything is enqueued; CUDA when a copy, a
 * launch or the synchronization fails (work before the failing step may
 * then have run).  Device status bits as for those calls. */
int qmla_decode_step(int format, void* blocks, int64_t num_blocks,
                     const int32_t* block_table, int32_t max_blocks_per_seq,
                     int32_t* seq_lens, int32_t max_seq_len, int32_t batch, int32_t heads,
                     int32_t n_new, const void* h_in, float softmax_scale, void* h_out,
                     void* workspace, size_t workspace_bytes, int32_t* status_dev,
                     void* stream);

/* Synchronize `stream`, read *status_dev and return QMLA_OK if it is 0,
 * QMLA_ERR_DEVICE otherwise (QMLA_ERR_CUDA if the copy failed). */
int qmla_read_status(const int32_t* status_dev, void* stream);

/* Static description of an error code ("ok", "invalid argument", ...). */
const char* qmla_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* QMLA_H_ */
