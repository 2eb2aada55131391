/*
 * fa_gb300.h -- FlashAttention-2 forward pass for one NVIDIA GB300 (sm_103a).
 *
 * The operation (page "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy 与
 * TiledMMA", section 先看全局: S = Q K^T, P = softmax(S), O = P V; the running
 * state m_i, l_i, o~_i of section 教学配置; the online update of section
 * 沿 C fragment 做 Online Softmax; the O + softmax-LSE output contract of
 * section 与官方 FA2 比较时，先对齐契约):
 *
 *   for batch b < B, head h < H, query row i < S, key j < S:
 *     z_ij       = scale * sum_d Q[b,i,h,d] * K[b,j,h,d]
 *     visible(j) = (j <= i) if causal else true
 *     O[b,i,h,:] = sum_{visible j} softmax_j(z_i.) * V[b,j,h,:]
 *     LSE[b,h,i] = ln sum_{visible j} exp(z_ij)          (natural log)
 *
 * computed tile by tile with an online softmax so that the S x S scores never
 * reach device memory.  Products of Q K^T and P V run on the tcgen05 tensor
 * cores with fp32 accumulation in tensor memory; P is rounded to the input
 * type before the second product; the row sum uses the unrounded fp32 P.
 *
 * Memory layout (all buffers are caller-owned DEVICE memory):
 *   Q, K, V, O : contiguous [B, S, H, D], element type fp16 or bf16 (all four
 *                the same), D a multiple of 8 from 8 to 256; base addresses
 *                16-byte aligned.  D = 64, 128, 192 and 256 run at full
 *                width; any other D runs on the next kernel up (the page
 *                "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy 与
 *                TiledMMA" lists other head dimensions among a production
 *                FA2's needs, section 哪些结论可以迁移，哪些只是本例特例): its
 *                tensor maps cover only the D columns, so the copies read the
 *                rest as zeros and the O stores leave it out, and the tensor
 *                cores do that padded work (a D = 96 call costs a D = 128 one).
 *                D > 128 has a kernel of its own (one 128-row query tile per
 *                CTA, 192 or 256 columns wide): the plain and grouped-K/V calls take it (the split
 *                entry points divide every tile's keys into the same number
 *                of chunks when the tiles fill less than three quarters of
 *                the SMs), and so do the packed, windowed and dropout
 *                calls (unsplit).
 *   LSE        : contiguous fp32 [B, H, S], or NULL to skip writing it.
 *
 * Ownership and ordering: the library keeps no pointer after a call returns
 * and allocates no device memory.  Work is enqueued on `stream` (0 = the
 * legacy default stream) and the call returns without waiting for it; the
 * caller orders any use of O / LSE after the stream.
 *
 * Errors: every entry point validates its arguments before launching and
 * returns an fa_status_t.  Nothing is launched when the status is not FA_OK.
 *   FA_ERR_INVALID_ARG  a NULL Q/K/V/O, B/H/S < 1, scale not finite or <= 0,
 *                       an unknown dtype, or sizes whose element count
 *                       overflows 64 bits
 *   FA_ERR_UNSUPPORTED  D not a multiple of 8 in [8, 256], a base address not 16-byte
 *                       aligned, ceil(S / 256) > 65535, or
 *                       B * H * ceil(S / 256) > 2^31 - 1
 *   FA_ERR_CUDA         a CUDA runtime or driver call failed (the CUDA error
 *                       is left set for the caller to read)
 *   FA_ERR_TIMEOUT      reported by fa_device_status() and
 *                       fa_last_device_status(): a device-side wait
 *                       exceeded its time limit and the kernel returned early
 *                       (the outputs of that call are undefined)
 *   FA_ERR_BAD_SEQLENS  reported by fa_device_status() and
 *                       fa_last_device_status(): fa_fwd_varlen found a
 *                       sequence offset out of range; nothing of that
 *                       sequence was read or written (its O / LSE rows are
 *                       left as they were)
 *   FA_ERR_DEVICE_CHECK reported by fa_device_status() and
 *                       fa_last_device_status() of a library built with
 *                       FA_DEBUG = 1 only: a device-side invariant check
 *                       failed (work-item bounds, the tensor-memory
 *                       allocation, the tile counts of the kernel's roles,
 *                       a stored row's sum); the kernel does not trap
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,
    FA_ERR_UNSUPPORTED = 2,
    FA_ERR_CUDA = 3,
    FA_ERR_TIMEOUT = 4,
    FA_ERR_BAD_SEQLENS = 5,
    FA_ERR_DEVICE_CHECK = 6
} fa_status_t;

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype_t;

/*
 * Forward pass on fp16 tensors.  Q, K, V, O: [B, S, H, D] fp16 device
 * pointers; LSE: [B, H, S] fp32 device pointer or NULL; causal: 0 or non-zero
 * (key j visible to query i iff j <= i); scale: finite, > 0 (1/sqrt(D) is the
 * usual choice).  Returns an fa_status_t.
 */
int fa_fwd_f16(const void* Q, const void* K, const void* V, void* O, float* LSE,
               int B, int H, int S, int D, int causal, float scale,
               fa_stream_t stream);

/* The same on bf16 tensors. */
int fa_fwd_bf16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                int B, int H, int S, int D, int causal, float scale,
                fa_stream_t stream);

/* The same with the element type passed as an fa_dtype_t value. */
int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
           int B, int H, int S, int D, int causal, float scale, int dtype,
           fa_stream_t stream);

/*
 * Split over keys (for shapes whose B * H * ceil(S / 256) query blocks leave
 * SMs idle: less than three quarters of a wave, or one to four waves with a
 * ragged last one).  The keys of some or all query blocks are divided among
 * several CTAs; each writes a partial result (unnormalised fp32 output rows,
 * the row max and the row sum) to `workspace`, and a second kernel, launched
 * on the same stream as a programmatic dependent of the first, merges them
 * with the same exp(m_old - m_new) rescaling that the online softmax uses
 * across key tiles (page "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy
 * 与 TiledMMA", section 沿 C fragment 做 Online Softmax).  Which blocks are
 * split, and how many ways, is fixed per shape (fa_split_plan).
 *
 * fa_splitkv_workspace_size: bytes of device workspace fa_fwd_splitkv needs
 * for this shape on the current device (0 when the shape is not split).
 * fa_splitkv_launches: kernels one fa_fwd_splitkv call launches (1 or 2; 0
 * for invalid sizes).
 * fa_fwd_splitkv: as fa_fwd, plus a caller-owned device workspace of
 * workspace_bytes bytes (16-byte aligned; may be NULL when the size query
 * returned 0).  Its contents need no initialisation and are overwritten.
 * Calls that share a workspace must be ordered on one stream.  Returns
 * FA_ERR_INVALID_ARG when the workspace is missing or too small.
 */
int fa_splitkv_workspace_size(int B, int H, int S, int D, int causal, size_t* bytes);
int fa_splitkv_launches(int B, int H, int S, int D, int causal);

/*
 * The split plan fa_fwd_splitkv uses for a shape on a GPU with `sms` SMs
 * (host only; no CUDA call).  splits[qb] receives the number of CTAs that
 * share the keys of query block qb (256 query rows; blocks 0 .. nblocks-1,
 * nblocks = ceil(S / 256)), for qb < min(nblocks, max_blocks); *items_per_head
 * (may be NULL) the work items of one head.  Returns the largest entry
 * (1 = not split), or FA_ERR_INVALID_ARG for sizes below 1 or a NULL
 * `splits` with max_blocks > 0.  Not part of the attention computation; the
 * pages have no counterpart.
 */
int fa_split_plan(int B, int H, int S, int D, int causal, int sms, int* splits, int max_blocks,
                  int* items_per_head);
int fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                   int B, int H, int S, int D, int causal, float scale, int dtype,
                   void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Grouped K/V heads (GQA; MQA when H_kv = 1).  The page "CuTe 详解：以
 * FlashAttention-2 拆解 Layout、TiledCopy 与 TiledMMA" lists GQA/MQA among
 * what a production FA2 forward also handles (section 哪些结论可以迁移，哪些只是
 * 本例特例); it gives no formula, and the reading here is the usual one:
 * K and V have H_kv heads, H_kv divides H, and query head h attends with
 * K/V head h / (H / H_kv) (consecutive query heads share a K/V head).
 *
 *   Q, O  [B, S, H, D] 16-bit, device       LSE [B, H, S] fp32 or NULL
 *   K, V  [B, S, H_kv, D] 16-bit, device    everything else as fa_fwd
 *
 * fa_fwd_gqa_splitkv splits the keys like fa_fwd_splitkv; its workspace size
 * is fa_splitkv_workspace_size(B, H, S, D, causal) (it does not depend on
 * H_kv).  Errors: as fa_fwd; FA_ERR_INVALID_ARG also when H_kv < 1 or H_kv
 * does not divide H.  fa_fwd(...) is fa_fwd_gqa(..., H_kv = H, ...).
 */
int fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE,
               int B, int H, int H_kv, int S, int D, int causal, float scale, int dtype,
               fa_stream_t stream);
int fa_fwd_gqa_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                       int B, int H, int H_kv, int S, int D, int causal, float scale,
                       int dtype, void* workspace, size_t workspace_bytes,
                       fa_stream_t stream);

/*
 * Test support: runs the forward (B = H = 1, non-causal) with the first
 * query tile's load withheld, so that the waits on it can never complete.
 * Every such wait gives up after about a second and the kernel ends early;
 * fa_device_status() then reports FA_ERR_TIMEOUT and the CUDA context stays
 * usable.  O is left undefined.  Errors before launch as fa_fwd.  Not part of
 * the attention computation; the pages have no counterpart.
 */
int fa_selftest_timeout(const void* Q, const void* K, const void* V, void* O, int S, int D,
                        int dtype, fa_stream_t stream);

/*
 * Attention dropout.  The page "CuTe 详解：以 FlashAttention-2 拆解 Layout、
 * TiledCopy 与 TiledMMA" lists dropout among what a production FA2 forward
 * also handles (section 哪些结论可以迁移，哪些只是本例特例) without a formula;
 * the reading here is the usual inverted dropout: each probability P_ij of
 * head (b, h) is kept with probability 1 - p_drop and the kept ones are scaled
 * by 1 / (1 - p_drop) before they multiply V.  The max, the row sums and LSE
 * are those of the undropped softmax.
 *
 * The mask is a pure function of (seed, b, h, i, j).  Each 32-bit word of a
 * Philox4x32-10 block (Salmon et al., "Parallel random numbers: as easy as
 * 1, 2, 3", SC 2011) holds two 16-bit draws, low half first; element
 * (b, h, i, j) takes draw j mod 8 (half j mod 2 of word (j mod 8) / 2) of the
 * block with counter (j / 8, i, h, b) and key (seed mod 2^32, seed / 2^32),
 * and is kept iff that draw >= floor(p_drop * 2^16) (so the keep probability
 * is within 2^-16 of 1 - p_drop).  p_drop = 0 keeps everything and gives
 * fa_fwd_gqa's result bit for bit.  Arguments and layout as fa_fwd_gqa (LSE may be NULL); the keys are not
 * split over CTAs.  Errors: as fa_fwd_gqa, and FA_ERR_INVALID_ARG unless
 * 0 <= p_drop < 1.
 */
int fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* LSE,
                   int B, int H, int H_kv, int S, int D, int causal, double p_drop,
                   unsigned long long seed, float scale, int dtype, fa_stream_t stream);

/*
 * Local (sliding-window) attention.  The page "CuTe 详解：以 FlashAttention-2
 * 拆解 Layout、TiledCopy 与 TiledMMA" names a "causal/local mask" among what a
 * production FA2 forward also handles (section 哪些结论可以迁移，哪些只是本例
 * 特例) without a formula; the reading here is the usual one: key j is kept
 * for query i iff i - window_left <= j <= i + window_right, -1 meaning no
 * bound on that side, and the causal mask caps the right bound at 0.  Key
 * tiles outside every row's window of a query tile are neither loaded nor
 * multiplied.  Arguments and layout as fa_fwd_gqa; the keys are not split
 * over CTAs.  Errors: as fa_fwd_gqa, and FA_ERR_INVALID_ARG for a window
 * bound below -1.
 */
int fa_fwd_local(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 int B, int H, int H_kv, int S, int D, int causal, int window_left,
                 int window_right, float scale, int dtype, fa_stream_t stream);

/*
 * Variable-length batch: B sequences packed along the token axis.  The page
 * "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy 与 TiledMMA" lists
 * variable-length sequences (变长序列) among what a production FA2 forward
 * also handles (section 哪些结论可以迁移，哪些只是本例特例) without a formula;
 * the reading here is the usual one: sequence b is rows
 * cu_seqlens[b] .. cu_seqlens[b+1]-1 of the packed tensors and attends only
 * within itself (causal positions count from the sequence start).
 *
 *   Q, O        [total, H, D] 16-bit, device
 *   K, V        [total, H_kv, D] 16-bit, device (H_kv divides H)
 *   LSE         [H, total] fp32, device, or NULL
 *   cu_seqlens  [B + 1] int32, device: cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[B] <= total, every length <= max_seqlen; read by
 *               the kernel (a sequence that breaks this is skipped and
 *               reported as FA_ERR_BAD_SEQLENS by fa_device_status())
 *   max_seqlen  the longest sequence (sizes the grid), 1 <= max_seqlen <= total
 *
 * Errors before launch: as fa_fwd (on one batch of `total` rows), and
 * FA_ERR_INVALID_ARG for a NULL cu_seqlens, B < 1, max_seqlen out of range
 * or H_kv not dividing H; FA_ERR_UNSUPPORTED for a cu_seqlens pointer that is
 * not 4-byte aligned.  The keys are not split over CTAs.
 */
int fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                  const int* cu_seqlens, int B, int max_seqlen, int total, int H, int H_kv,
                  int D, int causal, float scale, int dtype, fa_stream_t stream);

/*
 * fa_fwd_splitkv without a workspace argument, for callers that cannot
 * allocate device memory (for example a latency-critical loop that must not
 * pay for cudaMalloc's implicit device synchronisation, or a program whose
 * device memory belongs to an allocator it cannot reach from this call site).
 * The paper has no counterpart; it is a packaging of the split-over-keys path.
 *
 * The scratch is one device array inside this library, 24 MiB (25,165,824
 * bytes), reserved on every GPU that loads the library until the process
 * exits.  This call allocates nothing and calls no allocating routine.
 *   - It splits only the shapes whose query blocks fill less than three
 *     quarters of a wave (the one-wave plans); shapes that fa_fwd_splitkv
 *     would split over several waves run unsplit here, with the same result.
 *   - A shape whose one-wave split needs more than 24 MiB (what
 *     fa_splitkv_workspace_size reports for it, since such shapes are never
 *     multi-wave) is rejected with FA_ERR_UNSUPPORTED before anything is
 *     launched; shapes
 *     that are not split need no scratch and always run.  On a 152-SM GB300
 *     every split of D <= 64, and of D <= 128 without the causal mask, fits
 *     (at most about 20 MiB); the longest causal splits of 64 < D <= 128 (up
 *     to about 38 MiB, e.g. B = H = 1, S = 4096) are rejected.  Every split
 *     of D > 128 fits (at most one CTA per SM, 132 KiB of partials each).
 *   - The first call on a device looks up the array's device address on that
 *     device (with it current); make that first call before any stream
 *     capture on the device.
 *   - Every call shares the array and it keeps the last call's contents.
 *     Nothing in it has to start at zero: each call writes every partial
 *     result it later reads.  Each device has its own copy; two calls on one
 *     device whose work overlaps on the GPU (for example, issued on two
 *     streams) race on it and give undefined results: order them on one
 *     stream.
 * Arguments, layouts and the other status codes are those of fa_fwd.
 */
int fa_fwd_splitkv_static(const void* Q, const void* K, const void* V, void* O, float* LSE,
                          int B, int H, int S, int D, int causal, float scale, int dtype,
                          fa_stream_t stream);

/* Static text for a status code (never NULL). */
const char* fa_status_string(int status);

/*
 * Device-side status of the calls made so far on the current device:
 * FA_OK, or the first failure seen: FA_ERR_TIMEOUT if some kernel gave up on
 * a wait, FA_ERR_BAD_SEQLENS if fa_fwd_varlen met offsets out of range.  Synchronises
 * the device.  clear != 0 resets the word to FA_OK.  Returns FA_ERR_CUDA if the
 * status word cannot be read.
 */
int fa_device_status(int clear);

/*
 * The device status word as the calls enqueued on `stream` so far left it:
 * the word is read after all of that work (a copy ordered on `stream`, then a
 * wait for `stream` alone; other streams keep running).  Returns FA_OK,
 * FA_ERR_TIMEOUT or FA_ERR_BAD_SEQLENS as fa_device_status does, without
 * clearing it; FA_ERR_CUDA if the copy or the wait fails.  The word is one per
 * device (the current one) and shared by every stream on it, so a failure of
 * a kernel on another stream that finished before the read shows here too.
 * Do not call it inside a stream capture (it waits on the stream).
 */
int fa_last_device_status(fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
