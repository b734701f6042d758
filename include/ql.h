/*
 * libql - single-token decode of a dense Qwen3-style transformer with q4_0 weights and a
 * paged f16 KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * C ABI. Every entry point returns an int status (QL_OK = 0 or a negative QL_E* code) and
 * never throws. On failure ql_last_error() returns a thread-local message.
 *
 * Memory: every pointer named d_* is a DEVICE pointer owned by the caller; h_* / plain
 * pointers in the codec are HOST pointers. The library never frees caller memory. A model
 * handle owns only its own workspace (activation scratch, RoPE tables, attention partials,
 * captured graphs) and frees it in ql_model_destroy. Caller buffers must stay alive while any
 * call, handle or captured graph that references them may still run.
 *
 * Streams: kernel entry points are asynchronous on the given stream (a cudaStream_t passed as
 * void*, NULL = the legacy default stream). A returned QL_OK means the arguments validated and
 * the kernels were enqueued. Out-of-range indices found ON THE DEVICE (a block id outside the
 * pool, a position past the block table, a token outside the vocabulary) do not fault: the
 * kernel skips the access and records the first such event in a per-device error record that
 * ql_check_device_error() reads (it synchronizes the device).
 *
 * The first call on a device allocates that device's error record with cudaMalloc; make it
 * outside any stream capture (ql_model_create does it).
 *
 * Sources (public web pages; cited by page and item):
 *   [IL]  inferencelayer, src/cuda_llm.rs        - Q4Dev, CudaQwen3::{gemv, rms_add, step,
 *                                                   capture, run_graph}, rope_inv_freq
 *   [FK]  ferrum-kernels, backend/cuda/cuda_decode.rs - launch_paged_decode_attention,
 *                                                   attention_paged, alloc_block,
 *                                                   decode_step, batch_decode_step
 *   [ME]  memra-engine, qwen4exp_gpu.rs          - host_rms_norm, host_rope_at
 */
#ifndef QL_H
#define QL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
enum {
    QL_OK = 0,
    QL_EINVAL = -1,  /* bad argument (null pointer, bad shape, unsupported size)            */
    QL_ENOMEM = -2,  /* the library could not allocate its own workspace                     */
    QL_ECUDA = -3,   /* a CUDA launch or runtime call failed (message in ql_last_error)     */
    QL_EPOOL = -4,   /* KV block pool exhausted ([FK] alloc_block)                           */
    QL_ERANGE = -5,  /* an index is out of range (host-side check)                           */
    QL_EDEVICE = -6, /* a kernel recorded an out-of-range index (see ql_check_device_error) */
    QL_ESTATE = -7   /* call out of order, e.g. a graph replay before its capture            */
};

enum { QL_DTYPE_F32 = 0, QL_DTYPE_F16 = 1 };

/* GEMV epilogues */
enum {
    QL_EPI_NONE = 0,         /* y = W x                                                      */
    QL_EPI_ADD_RESIDUAL = 1, /* y = residual + W x (f32; y may be the residual buffer itself) */
    QL_EPI_SILU_MUL = 2      /* W = [gate | up] rows; y[b][i] = silu(g_i) * u_i, i < rows/2   */
};

const char* ql_status_str(int status);
const char* ql_last_error(void);
int ql_version(void);

/* --------------------------------------------------------------- q4_0 codec (host)
 * [IL] Q4Dev: a [rows, cols] matrix in 32-weight blocks; one f16 scale d and 16 bytes of
 * 4-bit codes q per block; weight = (q - 8) * d. Scales and codes are separate arrays,
 * row-major: scales [rows][cols/32] (f16 bit patterns), quants [rows][cols/32][16].
 * Byte j of a block holds element j in its low nibble and element j+16 in its high nibble.
 * Quantiser (the page does not print one; this is the rule the library fixes):
 *   d = nearest f16 (ties to even) of max|x|/7, computed in f64;
 *   q = clamp(round_half_even(x/d), -7, 7) + 8 in f64; a block with d == 0 gets q = 8.
 * For blocks with a normal f16 scale this gives |x - (q-8) d| <= d/2 for every weight.
 * Returns QL_EINVAL if cols % 32 != 0, a pointer is NULL, a weight is not finite or a block
 * scale overflows f16. Deterministic; uses several host threads for large matrices.      */
int ql_q4_0_pack(const float* w, int64_t rows, int64_t cols, uint16_t* scales,
                 uint8_t* quants);
/* w[r][32j+e] = (q - 8) * d, exactly (f32 holds every such product). */
int ql_q4_0_unpack(const uint16_t* scales, const uint8_t* quants, int64_t rows,
                   int64_t cols, float* w);
/* The same quantiser on the GPU (bit-identical to ql_q4_0_pack): d_w f32 [rows][cols] ->
 * d_scales, d_quants. A non-finite weight or an f16 overflow of a scale is recorded in the
 * device error record (that block is written as d = 0, q = 8). Asynchronous on stream.   */
int ql_q4_0_pack_device(const float* d_w, int64_t rows, int64_t cols, void* d_scales,
                        void* d_quants, void* stream);

/* --------------------------------------------------------------- q4_0 GEMV
 * [IL] CudaQwen3::gemv: y[b][r] = sum_k dq(W)[r][k] * x[b][k].
 * d_scales / d_quants: the q4_0 matrix above (device). d_x: f16 [batch][cols].
 * d_y: [batch][rows] (QL_EPI_SILU_MUL: [batch][rows/2]) in y_dtype (f32 or f16;
 * QL_EPI_ADD_RESIDUAL requires f32). d_residual: f32 [batch][rows] for QL_EPI_ADD_RESIDUAL,
 * else ignored; it may equal d_y. cols % 32 == 0; rows even for QL_EPI_SILU_MUL;
 * 1 <= batch <= 64. d_quants and d_x must be 16-byte aligned, d_scales, d_y and d_residual
 * 4-byte aligned (QL_EINVAL otherwise). Products and sums are f32: codes 1024 + q are exact
 * f16 operands of the tensor-core MMA, the -8 offset is folded into the accumulator, and each
 * 32-weight block is scaled in f32. Batches above 8 run in passes of at most 8 columns.    */
int ql_gemv_q4_0(const void* d_scales, const void* d_quants, int64_t rows, int64_t cols,
                 const void* d_x, int64_t batch, void* d_y, int y_dtype, int epilogue,
                 const float* d_residual, void* stream);

/* --------------------------------------------------------------- q4_0 tile stream (GPU)
 * The layout that the batch 1-2 GEMV copies with bulk (TMA) copies: the rows in 16-row tiles
 * (silu != 0: tile i = gate rows 8i..8i+7 followed by the matching up rows rows/2 + 8i..),
 * each tile as cols/128 units of 1152 contiguous bytes: the codes of 4 blocks x 16 rows
 * ([block][row], 16 B each) then the 16 rows' 4 f16 scales (8 B per row). Rows past the
 * matrix are zero. An exact byte permutation of the q4_0 arrays. cols % 128 == 0; with silu,
 * rows is even. Bytes needed: ql_q4_0_stream_bytes (0 on a bad shape).                   */
int64_t ql_q4_0_stream_bytes(int64_t rows, int64_t cols, int silu);
/* Re-lay d_scales / d_quants (the q4_0 arrays above, device) into d_stream. d_quants and
 * d_stream 16-byte aligned, d_scales 8-byte aligned. Asynchronous on stream.              */
int ql_q4_0_stream_pack(const void* d_scales, const void* d_quants, int64_t rows, int64_t cols,
                        int silu, void* d_stream, void* stream);
/* [IL] CudaQwen3::gemv at batch 1-32 from the tile stream: y = epilogue(W x).
 * d_x: f16 [batch][cols], 16-byte aligned. epilogue QL_EPI_NONE: d_y f32 [batch][rows];
 * QL_EPI_ADD_RESIDUAL: d_y f32 [batch][rows], y += W x in place; QL_EPI_SILU_MUL (d_stream
 * packed with silu): d_y f16 [batch][rows/2]. Batch 1-2: the activations are taken to 16-bit
 * fixed point with one power-of-two scale per 32-element block (x_int = round(x 2^s), |x_int|
 * < 2^15, relative error at most 2^-15 of the block's largest value); the products of codes and
 * x_int and each block's sum are exact 32-bit integers (dp2a), the -8 offset is subtracted
 * exactly, and each block is scaled by its f16 scale and 2^-s and accumulated in f32. Batch 3-32 (needs cols in 128..896 or a multiple of 1024): the
 * tensor-core form (A = (q - 8) d rounded once to f16, f16 x, f32 products and sums), split
 * over K in windows of 1024 columns so that every weight byte is streamed once; each window's
 * f32 partial sums go to d_workspace and are added in window order (deterministic) before the
 * epilogue: by a second kernel or (tcgen05 form, selectable) inside the kernel by the CTA that
 * finishes a row block's last window (an atomic ticket per row block). d_workspace
 * (device, 256-byte aligned, at least ql_gemv_q4_0_stream_workspace_bytes) is caller-owned
 * scratch, ZERO-FILLED before its first use; every call leaves it valid for the next call of
 * any shape (the tickets re-armed), unless the device error record reports a failed wait, after
 * which it must be zero-filled again. Calls that run concurrently need separate workspaces.
 * It may be NULL at batch 1-2. One CTA per SM; its waits are bounded (2 s, then the device error
 * record says so). QL_EINVAL for other batches.                                             */
int ql_gemv_q4_0_stream(const void* d_stream, int64_t rows, int64_t cols, const void* d_x,
                        int64_t batch, void* d_y, int epilogue, void* d_workspace,
                        int64_t workspace_bytes, void* stream);
/* The q4_0 GEMM for a chunk of prompt tokens ([IL] cuda_llm.rs: prefill, which its module doc
 * runs as sequential decode and its GemmEx arm on bf16 copies of the weights): y =
 * epilogue(W x_t) for n_tokens tokens at once, from the tile stream copy (d_stream, as for
 * ql_gemv_q4_0_stream). d_x: f16 [n_tokens][cols], 16-byte aligned; epilogue and d_y as for
 * ql_gemv_q4_0_stream with n_tokens in place of batch. On the tcgen05 tensor cores: one CTA per
 * 128 rows x NT tokens (NT = 256 above 128 tokens, 128 above 32, else 32), the weights expanded
 * into tensor memory as (q - 8) d rounded once to f16, f16 activations, f32 products and sums
 * (each output one tensor-core accumulator over K: the result does not depend on the call).
 * Every weight byte is read once per NT tokens. No workspace (no split over K, which the
 * chunked prefill uses with a workspace of its own); waits are bounded (2 s, then the device
 * error record says so). cols % 128 == 0 (even rows with SiLU*up), 1 <= n_tokens <= 2^20.
 * Asynchronous on stream.                                                                  */
int ql_gemm_q4_0_stream(const void* d_stream, int64_t rows, int64_t cols, const void* d_x, int64_t n_tokens,
                        void* d_y, int epilogue, void* stream);
/* Activation form of the batch 1-2 GEMV, for this process (ql_gemv_q4_0_stream and the decode
 * step at batch 1-2; graphs keep the form they were captured with):
 *   QL_GEMV_ACT_INT16 (default) 16-bit fixed point with one power-of-two scale per 32-element
 *                     block (above); products and block sums exact (dp2a).
 *   QL_GEMV_ACT_INT8  [IL] CudaQwen3::absmax + gemv: one scale per activation vector, read from
 *                     xs = [max|x|, 1/max|x|]; codes q = round_half_even(x * (127 / max|x|)),
 *                     the division and the product each one f32 operation; the weights are
 *                     multiplied by q * max|x| / 127 with dp4a (products and block sums exact
 *                     in 32 bits). Each output then differs from the exact product by at most
 *                     sum_k |w_k| * max|x| / 254 plus f32 rounding: a coarser form (the
 *                     decode step's logits tolerance is not met at the 8B width), selectable
 *                     for speed. RMSNorm'd inputs take max|x w| times the norm scale as max|x|.
 * The initial form is QL_GEMV_ACT_INT8 when the environment sets QL_GEMV_ACT=int8. Returns the
 * previous form, or QL_EINVAL for an unknown one.                                          */
enum { QL_GEMV_ACT_INT16 = 0, QL_GEMV_ACT_INT8 = 1 };
int ql_set_gemv_activation_form(int form);
/* Workspace bytes ql_gemv_q4_0_stream needs at batch 3-32 for this shape on the current
 * device (the split depends on its SM count); 0 on a bad shape.                           */
int64_t ql_gemv_q4_0_stream_workspace_bytes(int64_t rows, int64_t cols, int silu);
/* Tensor-core form of the batch 3-32 GEMV, for this process (ql_gemv_q4_0_stream and the
 * decode step; graphs keep the form they were captured with):
 *   QL_BATCHED_MMA_SYNC  (default) warps issue mma.sync m16n8k16 on the dequantised weights;
 *   QL_BATCHED_TCGEN05   a producer lane streams the codes into a 16-stage shared-memory ring
 *                        (tensor-map copies), 16 warps write (q - 8) d into tensor memory
 *                        (tcgen05.st), one lane issues tcgen05.mma (kind::f16, M 128, N 32,
 *                        K 16) against the staged activations into double-buffered f32
 *                        accumulators, 4 warps drain them as partial sums, and the second
 *                        kernel adds the K windows (QL_TC_KERNEL_MERGE=1 in the environment: the
 *                        CTA finishing a row block's last window does, by ticket). Same results
 *                        as the mma.sync form up to f32 summation order; slower on the decode
 *                        step at batch 32 (the MMA issue rate at N = 32 is the limit).
 * The initial form is QL_BATCHED_TCGEN05 when the environment sets QL_BATCHED_TC=1. Returns
 * the previous form, or QL_EINVAL for an unknown one.                                     */
enum { QL_BATCHED_MMA_SYNC = 0, QL_BATCHED_TCGEN05 = 1 };
int ql_set_batched_gemv_form(int form);

/* --------------------------------------------------------------- quantised KV rows (host)
 * The quantised KV-cache rows of [ME] (the quantised-cache storage: q8_row_bytes /
 * q5_row_bytes, the Q8Q5 store, and the host twins host_quant_q8_row, host_deq_q8_rows,
 * host_quant_q5_row, host_deq_q5_rows): keys as q8_0, values as q5_1. A row of dim f32
 * values is cut into 32-element blocks, a ragged last block padded with zeros that take part
 * in its statistics; every step is an f32 operation, f16 conversions round to nearest even.
 *   q8_0, 34 B per block: f16 d (little-endian), 32 int8 codes. d = max|x| / 127,
 *     id = 1/d (0 when d == 0 or 1/d is not finite), code = clamp(rint(x id), -127, 127);
 *     decoded f32(d) * code.
 *   q5_1, 24 B per block: f16 d, f16 m, a 32-bit word (bit l = bit 4 of code l), 16 bytes
 *     (byte l: code l's low nibble, code l+16's in the high nibble). d = (max - min) / 31,
 *     code = clamp(rint((x - min) id), 0, 31), m = min (a zero minimum stored as +0);
 *     decoded fma(f32(d), code, f32(m)).
 * x: host f32 [rows][dim]; out / in: host bytes [rows][row bytes]. Quantising returns
 * QL_EINVAL for a NULL pointer, rows or dim <= 0, a non-finite value, or a scale or minimum
 * that overflows f16. Deterministic, single-threaded.                                     */
int64_t ql_kv_q8_0_row_bytes(int64_t dim);
int64_t ql_kv_q5_1_row_bytes(int64_t dim);
int ql_kv_quantize_q8_0(const float* x, int64_t rows, int64_t dim, uint8_t* out);
int ql_kv_dequantize_q8_0(const uint8_t* in, int64_t rows, int64_t dim, float* x);
int ql_kv_quantize_q5_1(const float* x, int64_t rows, int64_t dim, uint8_t* out);
int ql_kv_dequantize_q5_1(const uint8_t* in, int64_t rows, int64_t dim, float* x);
/* The same codecs on the GPU, bit-identical to the host ones (both run one set of block
 * routines): d_x device f32 [rows][dim], d_out / d_in device bytes [rows][row bytes],
 * asynchronous on the stream. A non-finite value, or a scale or minimum that overflows f16,
 * is recorded in the device error record (ql_check_device_error) and the block's bytes are
 * still written. QL_EINVAL for NULL pointers or rows / dim <= 0.                          */
int ql_kv_quantize_q8_0_device(const float* d_x, int64_t rows, int64_t dim, uint8_t* d_out,
                               void* stream);
int ql_kv_dequantize_q8_0_device(const uint8_t* d_in, int64_t rows, int64_t dim, float* d_x,
                                 void* stream);
int ql_kv_quantize_q5_1_device(const float* d_x, int64_t rows, int64_t dim, uint8_t* d_out,
                               void* stream);
int ql_kv_dequantize_q5_1_device(const uint8_t* d_in, int64_t rows, int64_t dim, float* d_x,
                                 void* stream);

/* --------------------------------------------------------------- paged decode attention
 * [FK] launch_paged_decode_attention / attention_paged, split-K over the context:
 *   out[b][h][:] = sum_{t < context_lens[b]} softmax_t(q[b][h] . K_t * scale) V_t
 * with K_t, V_t of kv head g = h / (n_heads / n_kv_heads), stored at physical block
 * block_tables[b][t / block_size], slot t % block_size.
 * d_q: f16 [batch][n_heads][head_dim]. d_k_pool, d_v_pool: f16
 * [num_blocks][n_kv_heads][block_size][head_dim] (one layer). d_block_tables: int32
 * [batch][max_blocks_per_seq]. d_context_lens: int32 [batch], each in
 * [1, max_blocks_per_seq * block_size] (0 is allowed and marks an idle slot: its output is
 * left untouched). d_out: f16 [batch][n_heads * head_dim].
 * head_dim in {64, 128}; block_size 16; n_heads % n_kv_heads == 0, group <= 8.
 * Alignment: d_k_pool and d_v_pool 16-byte, d_q and d_out 4-byte (QL_EINVAL otherwise; nothing
 * is launched). A length above max_blocks_per_seq * block_size, or a block id outside
 * [0, num_blocks), is skipped on the device and recorded in the device error record; the output
 * row of such a sequence is then undefined.
 * d_workspace: ql_paged_attn_workspace_bytes(...) bytes, ZERO-FILLED before its first use
 * (the kernels leave it zero-filled again for the next call); one workspace per stream.  */
size_t ql_paged_attn_workspace_bytes(int64_t batch, int n_heads, int n_kv_heads,
                                     int head_dim, int block_size,
                                     int64_t max_blocks_per_seq);
int ql_paged_attn_decode(const void* d_q, const void* d_k_pool, const void* d_v_pool,
                         const int32_t* d_block_tables, const int32_t* d_context_lens,
                         int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                         int block_size, int64_t max_blocks_per_seq, int64_t num_blocks,
                         float scale, void* d_out, void* d_workspace,
                         size_t workspace_bytes, void* stream);

/* Causal attention of a prefill chunk ([IL] prefill as sequential decode: token t of the chunk,
 * at position *d_position + t, attends keys 0 .. *d_position + t): d_q f16 [n_tokens][n_heads]
 * [head_dim] (normalised and rotated), the sequence's K/V rows for positions 0 ..
 * *d_position + n_tokens - 1 already in d_k_pool / d_v_pool (layout as ql_paged_attn_decode),
 * d_block_table int32 [max_blocks_per_seq] of the sequence, d_position int32 [1] (device). Each
 * K/V block is read once for all the chunk's tokens (the chunk's tokens x query heads of a kv head
 * are the MMA rows); the block table's splits are merged by a second kernel. d_out f16
 * [n_tokens][n_heads * head_dim]. d_workspace: ql_paged_attn_chunk_workspace_bytes, contents
 * need not be initialised. Tolerance as ql_paged_attn_decode. Block ids out of range are
 * recorded in the device error record and their keys skipped. 1 <= n_tokens <= 256.       */
size_t ql_paged_attn_chunk_workspace_bytes(int64_t n_tokens, int n_heads, int n_kv_heads, int head_dim);
int ql_paged_attn_chunk(const void* d_q, const void* d_k_pool, const void* d_v_pool, const int32_t* d_block_table,
                        const int32_t* d_position, int64_t n_tokens, int n_heads, int n_kv_heads, int head_dim,
                        int block_size, int64_t max_blocks_per_seq, int64_t num_blocks, float scale, void* d_out,
                        void* d_workspace, size_t workspace_bytes, void* stream);

/* The same attention without a caller-supplied workspace, for callers that cannot allocate
 * device memory: for example a plugin inside a host application whose own pool owns all
 * device memory, or a latency-critical loop that cannot afford cudaMalloc/cudaFree (they can
 * synchronise the device). The pages have no counterpart; this is a library convenience.
 * Arguments mean what they mean for ql_paged_attn_decode. The split-K scratch comes from a
 * fixed 8 MiB array compiled into the library (held by every GPU that loads the library until
 * the process exits); a shape whose scratch, as ql_paged_attn_workspace_bytes reports it,
 * exceeds 8 MiB is rejected with QL_EINVAL. Nothing is allocated: the first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device current, so
 * make that first call before any stream capture. Every call clears the part of the array
 * that must start at zero, then shares the rest with every other call: calls whose kernels
 * overlap on the GPU (two streams, or two host threads) race on it and must be serialised by
 * the caller. The alignment rules and the host-side checks are those of ql_paged_attn_decode
 * (a misaligned pointer is QL_EINVAL and nothing is launched). Out-of-range block ids or lengths
 * are skipped on the device and the output rows of those sequences are undefined; they are
 * recorded for ql_check_device_error only if another libql call already created this device's
 * record. The looked-up address is kept for the life of the process: do not use this entry
 * point on a device after cudaDeviceReset.                                                 */
int ql_paged_attn_decode_noalloc(const void* d_q, const void* d_k_pool, const void* d_v_pool,
                                 const int32_t* d_block_tables, const int32_t* d_context_lens,
                                 int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                                 int block_size, int64_t max_blocks_per_seq, int64_t num_blocks,
                                 float scale, void* d_out, void* stream);

/* --------------------------------------------------------------- quantised KV pool
 * [ME] the quantised-cache storage (Q8Q5 store; host_quant_q8_row / host_quant_q5_row): keys as
 * q8_0 rows (f16 d = max|x| / 127, codes round(x / d) in [-127, 127]) and values as q5_1 rows
 * (f16 d = (max - min) / 31, f16 m = min, codes round((x - min) / d) in [0, 31]), per 32-element
 * block, every step one f32 operation (the rule of ql_kv_quantize_q8_0 / _q5_1 above).
 * Layout: one record of ql_kvq_record_bytes(head_dim) = 29 * head_dim bytes per (physical
 * block, kv head), a layer's pool [num_blocks][n_kv][record]. A record holds the block's 16 key
 * rows and 16 value rows, each field in its own array, all starting on 16-byte boundaries:
 *   key codes int8 [16][hd] at 0; value nibbles u8 [16][hd/2] at 16 hd (per 32-element block,
 *   byte l = code l | code l+16 << 4); key scales f16 [16][hd/32] at 24 hd; value bit 4 u32
 *   [16][hd/32] at 25 hd (bit l = code l's); value scales f16 [16][hd/32] at 27 hd; value minima
 *   f16 [16][hd/32] at 28 hd.
 * The page's q8_0 block is (key scale, 32 key codes), its q5_1 block (scale, minimum, bit-4
 * word, 16 nibble bytes): the same bytes in another order. head_dim 64 or 128 (0 otherwise).  */
int64_t ql_kvq_record_bytes(int head_dim);
/* Quantise d_k / d_v (f32 [n][n_kv_heads][head_dim], device) into one layer's pool: row i of kv
 * head g goes to slot d_slots[i] % 16 of the record of physical block d_slots[i] / 16
 * (int64 [n], device). A slot outside the pool is skipped and recorded in the device error
 * record, as is a non-finite value or an f16 overflow of a scale (the row is still written).
 * d_pool 16-byte aligned. Asynchronous on stream.                                          */
int ql_kvq_write(const float* d_k, const float* d_v, const int64_t* d_slots, int64_t n, int n_kv_heads,
                 int head_dim, void* d_pool, int64_t num_blocks, void* stream);
/* ql_paged_attn_decode over a quantised pool (d_pool: one layer, the layout above, 16-byte
 * aligned): keys and values are decoded as f16(d * code) and f16(fma(d, code, m)) and enter
 * the same split-K attention (ticket merge). Arguments, workspace and errors as for
 * ql_paged_attn_decode.                                                                     */
int ql_paged_attn_decode_kvq(const void* d_q, const void* d_pool, const int32_t* d_block_tables,
                             const int32_t* d_context_lens, int64_t batch, int n_heads, int n_kv_heads,
                             int head_dim, int block_size, int64_t max_blocks_per_seq, int64_t num_blocks,
                             float scale, void* d_out, void* d_workspace, size_t workspace_bytes,
                             void* stream);

/* How the context splits of a (sequence, kv head) are merged, for this process (every
 * attention entry point and the decode step; graphs keep the form they were captured with).
 * Both forms take the same online-softmax merge over the splits in order, so their outputs
 * are bit-identical ([FK] split-K flash-decode reduce, [IL] attn_reduce):
 *   QL_ATTN_MERGE_TICKET  (default) each split writes its partial to the workspace and the
 *                         last one to take an atomic ticket merges them all; the others exit
 *                         at once, freeing their SMs for the next kernel.
 *   QL_ATTN_MERGE_CLUSTER the splits are one thread-block cluster; each keeps its
 *                         partial in shared memory and, after a cluster barrier, merges a
 *                         slice of the outputs from the others' partials through distributed
 *                         shared memory. Used at batch 1-2 with 2..16 splits when the device
 *                         can hold every cluster of the launch at once; otherwise the ticket.
 *                         Every split then lives until the merge ends (slower in the decode
 *                         step: the next kernel's CTAs wait for those SMs).
 * The initial form is QL_ATTN_MERGE_CLUSTER when the environment sets QL_ATTN_MERGE=1.
 * Returns the previous form, or QL_EINVAL for an unknown one.                              */
enum { QL_ATTN_MERGE_TICKET = 0, QL_ATTN_MERGE_CLUSTER = 1 };
int ql_set_attn_merge_form(int form);
/* The merge form an attention launch of this shape takes on the current device under the
 * current setting (QL_ATTN_MERGE_TICKET or QL_ATTN_MERGE_CLUSTER), or a negative QL_E* code
 * (QL_EINVAL for a shape the attention rejects).                                           */
int ql_paged_attn_merge_form(int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                             int64_t max_blocks_per_seq);

/* --------------------------------------------------------------- qk-norm + RoPE + KV append
 * [IL] CudaQwen3::step (qk_norm_rope kernel), [FK] decode_step / attention_paged:
 * for slot b at position p = d_positions[b]:
 *   q_h = rope(rms(q_h) * q_norm, p), k_g = rope(rms(k_g) * k_norm, p)  (RMS over head_dim,
 *   [ME] host_rms_norm), V unchanged; rope is the NeoX split-half rotation of pairs
 *   (i, i + head_dim/2) by angle p * theta^(-2i/head_dim) ([ME] host_rope_at,
 *   [IL] rope_inv_freq), taken from the tables d_cos/d_sin [max_position][head_dim/2].
 * d_qkv: f32 [batch][(n_heads + 2 n_kv_heads) * head_dim] (rows q | k | v).
 * Writes q as f16 [batch][n_heads][head_dim] to d_q_out and K, V (f16) to pool slot
 * (block_tables[b][p / block_size], p % block_size) of kv head g.
 * d_active: int32 [batch] or NULL; a slot with active == 0 is skipped.                    */
int ql_fused_norm_rope(const float* d_qkv, const float* d_q_norm_w, const float* d_k_norm_w,
                       const float* d_cos, const float* d_sin, const int32_t* d_positions,
                       const int32_t* d_active, float eps, int64_t batch, int n_heads,
                       int n_kv_heads, int head_dim, void* d_q_out, void* d_k_pool,
                       void* d_v_pool, const int32_t* d_block_tables,
                       int64_t max_blocks_per_seq, int block_size, int64_t num_blocks,
                       int64_t max_position, void* stream);
/* Host: cos/sin tables [max_position][head_dim/2] (f32, computed in f64) for theta. */
int ql_rope_tables(float* h_cos, float* h_sin, int64_t max_position, int head_dim,
                   double theta);

/* --------------------------------------------------------------- model + decode step */
typedef struct {
    const void* scales; /* f16 [rows][cols/32] (device) */
    const void* quants; /* u8  [rows][cols/32][16] (device) */
    int64_t rows, cols;
} ql_q4_0_matrix;

typedef struct {
    const float* attn_norm; /* [hidden] */
    const float* ffn_norm;  /* [hidden] */
    const float* q_norm;    /* [head_dim] */
    const float* k_norm;    /* [head_dim] */
    ql_q4_0_matrix qkv;     /* [(n_heads + 2 n_kv) * head_dim, hidden], rows q | k | v */
    ql_q4_0_matrix o;       /* [hidden, n_heads * head_dim] */
    ql_q4_0_matrix gate_up; /* [2 * intermediate, hidden], rows gate | up (dense models) */
    ql_q4_0_matrix down;    /* [hidden, intermediate] (dense models) */
    /* routed experts (num_experts > 0; [IL] Cfg and the MoE weights as loaded): */
    const float* router;             /* f32 [num_experts][hidden] */
    ql_q4_0_matrix experts_gate_up;  /* [num_experts * 2 * moe_inter, hidden]: expert e owns rows
                                        [e 2mi, e 2mi + mi) (gate) and the next mi (up)     */
    ql_q4_0_matrix experts_down;     /* [num_experts * hidden, moe_inter]: expert e owns rows
                                        [e hidden, (e + 1) hidden)                         */
} ql_layer_desc;

typedef struct {
    int64_t hidden, n_layers, n_heads, n_kv_heads, head_dim, intermediate, vocab;
    float eps;                  /* RMSNorm epsilon */
    double rope_theta;
    const float* embed;         /* f32 [vocab][hidden] (device) */
    const float* final_norm;    /* [hidden] */
    ql_q4_0_matrix lm_head;     /* [vocab, hidden] (untied) */
    const ql_layer_desc* layers;/* HOST array [n_layers] of device pointers; copied */
    void* k_pool;               /* f16 [n_layers][num_blocks][n_kv][block_size][head_dim] */
    void* v_pool;               /* same */
    int64_t num_blocks;
    int block_size;             /* 16 */
    int64_t max_batch;          /* largest batch any step will use */
    int64_t max_blocks_per_seq; /* block-table row length; max context = this * block_size */
    int kv_format;              /* QL_KV_F16 (k_pool / v_pool) or QL_KV_Q8_0_Q5_1 (kvq_pool) */
    void* kvq_pool;             /* QL_KV_Q8_0_Q5_1: u8 [n_layers][num_blocks][n_kv][ql_kvq_record_bytes] */
    /* Routed experts ([IL] Cfg: num_experts, topk, moe_inter, norm_topk; 0 experts = dense).
     * Every layer's feed-forward block is then: router logits = router . rms(x) w_ffn (f32),
     * the softmax over all experts, the topk largest (lowest index first on ties), their weights
     * renormalised to sum 1 when norm_topk; per selected expert silu(gate) * up and its down
     * rows; x += the weighted sum in slot order. Decode steps at batch 1 only (QL_EINVAL for a
     * larger batch); intermediate, gate_up and down are then unused. moe_inter and hidden must
     * be multiples of 128, num_experts <= 512, topk <= 64.                                    */
    int64_t num_experts, topk, moe_inter;
    int norm_topk;
} ql_model_desc;

/* KV cache formats of a model (ql_model_desc.kv_format). QL_KV_Q8_0_Q5_1: the quantised pool of
 * ql_paged_attn_decode_kvq; the decode step quantises each appended K row as q8_0 and V row as
 * q5_1 (ql_kvq_write's rule) and reads every record back through the quantised attention. The
 * persistent step kernel takes only QL_KV_F16.                                            */
enum { QL_KV_F16 = 0, QL_KV_Q8_0_Q5_1 = 1 };

typedef struct ql_model ql_model;

/* Validates dims and allocates the handle's workspace on the current device. */
int ql_model_create(const ql_model_desc* desc, ql_model** out);
int ql_model_destroy(ql_model* m);

/* How a decode step runs. QL_STEP_LAUNCHES: one kernel per phase (q|k|v, attention, o,
 * gate|up, down per layer; lm_head), any batch up to max_batch; at batch 1-2 the GEMVs read
 * the tile stream copy of the weights (see ql_gemv_q4_0_stream). QL_STEP_PERSISTENT: the whole
 * step as ONE cooperative kernel, one CTA per SM, that streams every layer's weights through
 * shared-memory rings and separates the phases with grid-wide barriers in device memory;
 * batches up to ql_model_persistent_max_batch() (at most 2). QL_STEP_AUTO (the default):
 * QL_STEP_LAUNCHES, the faster of the two on GB300 (1.55 vs 2.89 ms per batch-1 step of the
 * 8B-shaped model). Both compute the same step ([IL] CudaQwen3::step); their sums differ only
 * in rounding order.                                                                     */
enum { QL_STEP_AUTO = 0, QL_STEP_LAUNCHES = 1, QL_STEP_PERSISTENT = 2 };
/* Options of a model handle:
 *   QL_OPT_STEP_KERNEL         one of QL_STEP_*; QL_STEP_PERSISTENT is QL_EINVAL when the
 *                              model has no persistent kernel (max batch 0)
 *   QL_OPT_BARRIER_TIMEOUT_NS  bound on every grid-barrier wait of the persistent step
 *                              (default 2e9 ns). A wait that runs out records a device error
 *                              (read with ql_check_device_error), every CTA leaves the step
 *                              and the step's outputs are not written; the next step runs
 *                              normally. Nothing else waits on another CTA.
 *   QL_OPT_TEST_BARRIER_EXTRA  0 (default) or 1: every barrier of the persistent step also
 *                              waits for one arrival that never comes, so the bounded wait
 *                              runs out (failure-path tests; no fault, the context stays usable)
 *   QL_OPT_STEP_TRACE          device address of a uint64 buffer of at least
 *                              (2 + 5 n_layers + 1) * num_SMs * 8 entries, or 0 (default, off):
 *                              the persistent step writes globaltimer stamps (ns) there as
 *                              [row][CTA][8]: row 0 entry 0/1 = the CTA's start; row k >= 1,
 *                              entries 0/1 = arrival at / exit from barrier k, entries 2..5 =
 *                              steps of the phase that ends at barrier k (GEMV: activations
 *                              staged, warp 0's units done, all warps done, epilogues done;
 *                              attention: q ready, blocks merged, split ticket taken, end).
 *                              A step of separate launches stamps its GEMV launches
 *                              instead (buffer: (5 n_layers + 1) * num_SMs * 8 entries): launch
 *                              k (qkv, o, gate_up, down of each layer, then lm_head) fills row
 *                              k, per CTA (at most num_SMs CTAs): 0 start,
 *                              1 predecessor done, 2 activations staged, 3 units done (batch
 *                              1-2: warp 0's), 4 all warps done / partial sums written, 5 end
 *                              (6, 7 at batch 1-2: warp 0's cycles waiting for bulk copies /
 *                              in its unit loop; else 0); the attention launch of layer l fills
 *                              row 4 n_layers + 1 + l for its first num_SMs CTAs: 0 start, 1
 *                              predecessor done, 2 q ready, 3 blocks done, 4 split ticket
 *                              taken, 5 end, 6 = 1 for the CTA that merged the splits. A
 *                              profiling aid
 *   QL_OPT_MERGE_TRACE         device address of a uint64 buffer of at least
 *                              (4 n_layers + 1) * num_SMs * 4 entries, or 0 (default, off):
 *                              at batch 3-32 the merge launch that adds up the K windows of
 *                              GEMV launch k (numbered as for QL_OPT_STEP_TRACE) fills row k,
 *                              per CTA (num_SMs CTAs): 0 start, 1 past its wait on the GEMV,
 *                              2 the CTA's outputs written, 3 end. Other batch sizes leave it
 *                              untouched. A profiling aid
 * Applies to steps issued (or graphs captured) afterwards. QL_EINVAL for anything else.  */
enum { QL_OPT_STEP_KERNEL = 1, QL_OPT_BARRIER_TIMEOUT_NS = 2, QL_OPT_TEST_BARRIER_EXTRA = 3,
       QL_OPT_STEP_TRACE = 4, QL_OPT_MERGE_TRACE = 5 };
int ql_model_set_option(ql_model* m, int option, int64_t value);
/* When the persistent kernel is available, ql_model_create also keeps a copy of every q4_0
 * matrix re-laid as a tile stream (16 rows x 4 blocks of codes and their scales contiguous,
 * 1152 B per unit) for the kernel's bulk copies: device memory equal to the weights again.
 * The weights must not change after ql_model_create.
 * Largest batch the persistent step kernel takes for this model on its device: 0 when the
 * shape or the device does not allow it (matrix widths must be multiples of 128, codes 16-byte
 * and scales 8-byte aligned, one CTA with ~200 KB of shared memory per SM).              */
int64_t ql_model_persistent_max_batch(const ql_model* m);

/* One decode step for `batch` slots ([IL] CudaQwen3::step, [FK] batch_decode_step).
 * Every per-step input lives in device memory so the step can be captured and replayed:
 *   tokens      int32 [batch]  this step's token per slot (read)
 *   positions   int32 [batch]  position of tokens[b]; its K/V is appended there and the
 *                              attention covers positions 0..positions[b]; advanced by one
 *                              for every active slot at the end of the step
 *   block_tables int32 [batch][max_blocks_per_seq] of the model; blocks for position
 *                              positions[b] must be assigned before the step
 *   active      int32 [batch] or NULL (all active); inactive slots append nothing, keep
 *                              their position and their next token
 *   logits      f32 [batch][vocab] or NULL (then kept in the workspace)
 *   next_tokens int32 [batch]  greedy argmax of the logits, lowest index on ties; may be
 *                              the tokens buffer itself (feeds the next replay)
 *   out_tokens  int32 [batch][out_stride] or NULL: next token also written at index
 *                              positions[b] + 1 (if < out_stride)                          */
typedef struct {
    int64_t batch;
    const int32_t* tokens;
    int32_t* positions;
    const int32_t* block_tables;
    const int32_t* active;
    float* logits;
    int32_t* next_tokens;
    int32_t* out_tokens;
    int64_t out_stride;
} ql_step_args;

int ql_decode_step(ql_model* m, const ql_step_args* args, void* stream);
/* Capture one ql_decode_step with these arguments as a CUDA graph keyed by args->batch
 * ([IL] CudaQwen3::capture). Replaces an earlier graph of the same batch.               */
int ql_decode_graph_capture(ql_model* m, const ql_step_args* args, void* stream);
/* Replay the graph of this batch n_steps times back to back ([IL] run_graph).
 * QL_ESTATE if no graph of that batch was captured.                                    */
int ql_decode_graph_replay(ql_model* m, int64_t batch, int n_steps, void* stream);
/* One decode step from host buffers: copies h_tokens (int32 [batch], host; pinned memory keeps
 * the copy asynchronous) into the tokens buffer the graph of this batch was captured with,
 * replays the graph once, copies its next_tokens buffer into h_next_tokens (int32 [batch],
 * host) and waits for the stream, so that h_next_tokens holds the step's greedy tokens on
 * return. h_tokens and h_next_tokens may be the same buffer (a greedy loop feeding each step's
 * tokens to the next): the copies are ordered on the stream. The other step buffers
 * (positions, tables, logits) stay on the device and advance as with ql_decode_graph_replay.
 * QL_ESTATE if no graph of that batch was captured.                                        */
int ql_decode_graph_step_host(ql_model* m, int64_t batch, const int32_t* h_tokens, int32_t* h_next_tokens,
                              void* stream);
/* Chunked prefill of one sequence. [IL] runs a prompt as sequential decode (its module doc);
 * here a chunk of n_tokens prompt tokens (d_tokens int32 [n_tokens], device) at positions
 * *d_position .. *d_position + n_tokens - 1 goes through every layer together: the GEMVs take
 * the chunk as their batch (every weight byte streamed once per chunk; the split-K tensor-core
 * form from 3 tokens; above 32 tokens the tcgen05 GEMM of ql_gemm_q4_0_stream, once per 256
 * tokens), qk-norm + RoPE append all its K/V rows to the sequence's blocks, then
 * each token attends causally to positions 0 .. its own. The result equals n_tokens decode
 * steps of those tokens (teacher-forced) up to rounding. d_block_table: int32
 * [max_blocks_per_seq] of the sequence (blocks for every position of the chunk assigned);
 * d_position: int32 [1], advanced by n_tokens; d_logits: f32 [vocab] of the chunk's last token,
 * or NULL; d_next_token: int32 [1], its greedy argmax, or NULL. 1 <= n_tokens <= min(256,
 * max_batch); dense models with the f16 KV format. Asynchronous on stream; not for capture. */
int ql_prefill_chunk(ql_model* m, const int32_t* d_tokens, int64_t n_tokens, int32_t* d_position,
                     const int32_t* d_block_table, float* d_logits, int32_t* d_next_token, void* stream);
/* Synchronizes the device and reads (and clears) its error record: QL_OK, or QL_EDEVICE
 * with the first recorded event described in ql_last_error(). m may be NULL.            */
int ql_check_device_error(ql_model* m);

/* --------------------------------------------------------------- KV block allocator (host)
 * [FK] alloc_block / release_kv_cache: take the most recently freed block first, else the
 * next never-used id; QL_EPOOL when the pool is exhausted.                               */
typedef struct ql_block_pool ql_block_pool;
int ql_block_pool_create(int64_t num_blocks, ql_block_pool** out);
int ql_block_pool_destroy(ql_block_pool* p);
int ql_block_pool_alloc(ql_block_pool* p, int32_t* out_id);
int ql_block_pool_free(ql_block_pool* p, const int32_t* ids, int64_t n);
int64_t ql_block_pool_in_use(const ql_block_pool* p);

#ifdef __cplusplus
}
#endif
#endif /* QL_H */
