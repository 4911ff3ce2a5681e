/*
 * dflash.h -- C ABI of the DFlash draft-and-verify hot path on GB300 (sm_103a).
 *
 * One DFlash cycle (page "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with
 * DFlash", section "The released serving cycle") is, on the drafter side:
 *   1. dflash_fuse_context  -- concatenate the captured target hidden states on
 *      the feature axis, project them to the draft width (W_c) with RMSNorm, and
 *      project that into K/V entries appended to every draft layer's cache
 *      (same page, "Five target states become persistent draft context";
 *      page "DFlash & DFlash2: Block-Diffusion LLM-Speedup", 4.1).
 *   2. dflash_block_attn    -- one non-causal attention of the draft block
 *      (anchor + mask positions) over the cached context plus the block, GQA,
 *      per-head Q/K RMSNorm before RoPE (E4B page, same section).
 *   3. dflash_verify        -- exact speculative verification: min(1, p/q)
 *      acceptance, a correction drawn from the normalised max(0, p - q)
 *      residual, or argmax matching under greedy decoding (E4B page, "Why exact
 *      verification preserves the target"; DFlash2 page, 4.4).
 * Beyond the cycle: the drafter's head and sampling (section 4), the rest of a
 * draft layer (section 5) and the DFlash2 variants (section 6).  The cache
 * descriptor takes a linear, ring (sliding window) or paged (block table)
 * layout.
 *
 * Conventions for every call
 *  - All tensor pointers are DEVICE pointers (cudaMalloc'd, or any memory the
 *    GPU can address), owned by the caller.  The library never allocates device
 *    memory; scratch space is the caller's `workspace` of at least the size the
 *    matching *_workspace_size() function returns (256-byte aligned).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls enqueue kernels on it and return without synchronising.
 *  - Every argument is validated on the host before any launch; on a non-zero
 *    status nothing has been enqueued and nothing is written.
 *  - Conditions only the device can see (a sequence whose seq_len + n_new
 *    exceeds the cache capacity, a draft token outside [0, V), a paged
 *    block-table entry outside the pool) never fault:
 *    the kernel skips the affected writes and raises a bit in the library's
 *    device status word, read with dflash_read_device_status().
 *  - Tensors are dense, row-major, in the stated shape.  One dtype per call:
 *    DFLASH_BF16 (storage bf16, float32 arithmetic) or DFLASH_F32.
 *  - Reading of positions (the pages do not fix them): cached context row t of
 *    a sequence sits at cache position t; block row j sits at seq_len[b] + j.
 *  - RoPE pairs element e with e + d/2 and turns it by pos * theta^(-2e/d).
 *  - Weight orientation: every weight is stored with its input (K) dimension
 *    contiguous.  W_c is taken as the DFlash2 page writes it (4.1), D rows of
 *    J * d_t, so Y = concat(taps) W_c^T; W_kv and the drafter's projections
 *    are [outputs][inputs] (the nn.Linear layout).  A [J * d_t, D] listing of
 *    W_c is this matrix transposed.
 *  - RoPE theta and the RMSNorm eps are plain float arguments of each call
 *    (1e6 and 1e-6 in the pages' drafter configuration), not a struct.
 *  - Status 5 is a workspace error (NULL, misaligned or too small); there is
 *    no debug-only status: conditions only the device sees are reported
 *    through the device status word in every build.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int dflash_status;
enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARGUMENT = 1, /* null pointer, negative size, bad alignment  */
  DFLASH_ERR_UNSUPPORTED = 2,      /* a shape or dtype the library does not handle */
  DFLASH_ERR_CAPACITY = 3,         /* host-visible size exceeds the cache capacity */
  DFLASH_ERR_CUDA = 4,             /* a CUDA call failed: dflash_last_error_string */
  DFLASH_ERR_WORKSPACE = 5         /* workspace NULL, misaligned or too small     */
};

typedef int dflash_dtype;
enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 };

/* Bits of the device status word (dflash_read_device_status). */
enum {
  DFLASH_DEV_CAPACITY = 1u << 0,   /* fuse_context: seq_len[b]+n_new[b] > capacity; rows skipped */
  DFLASH_DEV_BAD_TOKEN = 1u << 1,  /* verify: draft token outside [0, V); treated as rejected   */
  DFLASH_DEV_BAD_SEQLEN = 1u << 2, /* seq_len[b] < 0 or > capacity, or (paged) a block-table
                                      entry a new row needs outside [0, num_pages); row skipped */
  DFLASH_DEV_TIMEOUT = 1u << 3     /* a bounded wait inside a kernel gave up (never expected) */
};

/*
 * Draft KV cache, one per draft model (all layers).  Caller-owned.
 *   k, v    : linear: [num_layers][batch][num_kv_heads][capacity][head_dim];
 *             paged: [num_layers][num_pages][num_kv_heads][page_size][head_dim]
 *             (a page is page_size consecutive positions of one sequence, for
 *             every KV head and both K and V of the layer); dtype.
 *             K rows hold keys already RMS-normalised and rotated.
 *   seq_len : device int32 [batch], cached positions per sequence.  The calls
 *             read it and never advance it: after dflash_fuse_context the
 *             caller adds n_new[b] (rolling back a rejected proposal = not
 *             advancing; block K/V are never written to the cache).
 *   ring    : 0: position p is row p (seq_len <= capacity).  1: the cache is
 *             the draft's sliding window (E4B page, the released drafter's
 *             1024-token window): position p is row p % capacity, seq_len may
 *             exceed capacity, and attention sees the latest
 *             min(seq_len, capacity) positions (block_attn's window must be 0).
 *             A fusion call may add at most capacity rows per sequence.
 *   block_table : NULL for the linear layout.  Paged layout (the ragged
 *             serving shape: sequences take pages from a shared pool as they
 *             grow; E4B page "Cache and latency have separate break-even
 *             points" counts the cache payload before paging, DFlash2 page 7.2
 *             keeps the draft cache in a paged memory manager; neither fixes a
 *             layout, this one is the library's): device int32 [batch][max_pages]; position p of sequence b
 *             lives in page block_table[b * max_pages + p / page_size], row
 *             p % page_size.  capacity must equal max_pages * page_size;
 *             page_size a multiple of 128 (one attention key tile never
 *             crosses a page); bf16 only; ring must be 0; block_attn's window
 *             must be 0.  Entries past a sequence's length are never read; a
 *             needed entry outside [0, num_pages) raises DFLASH_DEV_BAD_SEQLEN
 *             and the fusion skips the row (attention reads zeros there).
 */
typedef struct {
  int num_layers;
  int batch;
  int num_kv_heads;
  int head_dim;    /* must be 128 */
  int capacity;    /* positions per (layer, sequence, head), >= 1 */
  dflash_dtype dtype;
  void* k;
  void* v;
  const int32_t* seq_len;
  int ring;        /* 0: linear cache, 1: ring buffer of capacity rows (sliding window) */
  const int32_t* block_table;  /* NULL: linear layout; else the paged layout's [batch][max_pages] */
  int page_size;   /* paged: positions per page (multiple of 128) */
  int num_pages;   /* paged: pages in the pool (the k/v arrays' second dimension) */
  int max_pages;   /* paged: block-table entries per sequence */
} dflash_kv_cache;

/* ---------------------------------------------------------------------------
 * 1. Context fusion and K/V injection.
 *    E4B page "Five target states become persistent draft context"; DFlash2
 *    page 4.1:  H_t = RMSNorm(W_c [H^(l1); ...; H^(lJ)]),  K_l = W_l^K H_t,
 *    V_l = W_l^V H_t.  Every key then gets the per-head RMSNorm (gain k_gain[l])
 *    and RoPE at its cache position before it is stored.
 *
 *  num_taps, taps : J device pointers (host array of J pointers), each
 *                   [total_new, d_target]; tap order = ascending target layer.
 *                   Rows are packed by sequence: rows cu_new[b] .. cu_new[b+1]-1
 *                   belong to sequence b.  16-byte aligned.
 *  cu_new         : device int32 [batch+1], cu_new[0] = 0, non-decreasing,
 *                   cu_new[batch] = total_new.
 *  w_fuse         : [d_model, J*d_target]   (W_c in the pages' orientation)
 *  g_fuse         : [d_model] RMSNorm gain (NULL = ones)
 *  w_kv           : [L*2*Hkv*128, d_model]; output column
 *                   ((l*2 + s)*Hkv + h)*128 + e, s = 0 key, 1 value
 *  k_gain         : [L, 128] per-layer key-norm gain (NULL = ones)
 *  rope_theta, eps: RoPE base (1e6 by default) and RMSNorm epsilon (1e-6)
 *  cache          : host pointer to the cache descriptor; K/V rows
 *                   seq_len[b] .. seq_len[b]+n_new[b]-1 of every layer are
 *                   written.  dtype of cache, taps and weights must agree.
 *  h_t_out        : optional [total_new, d_model] copy of H_t (may be NULL)
 * Constraints (bf16): d_target % 64 == 0, d_model % 256 == 0, head_dim 128.
 * Ownership: reads all inputs, writes cache rows, h_t_out and the workspace.
 * ------------------------------------------------------------------------- */
DFLASH_API size_t dflash_fuse_context_workspace_size(int total_new, int num_taps, int d_target, int d_model,
                                          int num_layers, int num_kv_heads, dflash_dtype dtype);

DFLASH_API dflash_status dflash_fuse_context(int num_taps, const void* const* taps, int d_target,
                                  const int32_t* cu_new, int batch, int total_new,
                                  const void* w_fuse, const void* g_fuse, int d_model,
                                  const void* w_kv, const void* k_gain,
                                  float rope_theta, float eps,
                                  const dflash_kv_cache* cache, void* h_t_out,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * 2. Draft-block attention of one layer.
 *    E4B page "The released serving cycle" (steps 2-3) and "Five target
 *    states...": Q [B,Hq,bs,128] and K/V [B,Hkv,bs,128] of the block,
 *    Hq/Hkv query heads per KV head, per-head Q/K RMSNorm before RoPE; the
 *    block attends to the cached context plus itself, non-causally.
 *
 *  layer        : draft layer index into the cache (0 .. L-1)
 *  batch, block_size, num_q_heads : B, bs (1..16), Hq (Hq % Hkv == 0,
 *                 Hq/Hkv * bs <= 64)
 *  q            : [B, Hq, bs, 128]    kb, vb : [B, Hkv, bs, 128]
 *                 (q, kb, vb and out 16-byte aligned: the rows are loaded
 *                 and stored in bulk; else status 1 and nothing enqueued)
 *  q_gain, k_gain: [128] this layer's norm gains (NULL = ones)
 *  window       : 0 = the whole cached context, else the latest `window`
 *                 cached positions
 *  out          : [B, Hq, bs, 128] = softmax(q^ K^T / sqrt(128)) V with
 *                 q^ = RoPE(RMSNorm(q) * q_gain) at position seq_len[b]+j and
 *                 keys = cache[layer][b][h/(Hq/Hkv)][lo..seq_len[b]) ++
 *                 RoPE(RMSNorm(kb) * k_gain).
 * bf16 rounding points: q^ and the block keys (before the products) and out.
 * The workspace holds the split partials and the call's counters (cleared by
 * the call itself): two calls in flight at once need two workspaces.
 * ------------------------------------------------------------------------- */
DFLASH_API size_t dflash_block_attn_workspace_size(int batch, int block_size, int num_q_heads,
                                        int num_kv_heads, int capacity, int window,
                                        dflash_dtype dtype);

DFLASH_API dflash_status dflash_block_attn(int layer, int batch, int block_size, int num_q_heads,
                                const void* q, const void* kb, const void* vb,
                                const void* q_gain, const void* k_gain,
                                float rope_theta, float eps,
                                const dflash_kv_cache* cache, int window,
                                void* out, void* workspace, size_t workspace_bytes,
                                void* stream);

/* ---------------------------------------------------------------------------
 * 3. Exact speculative verification.
 *    E4B page "Why exact verification preserves the target"; DFlash2 page 4.4
 *    (acceptance, residual, greedy rule) and FAQ Q3 (temperature).
 *
 *  target_logits : [B, bs, V]; row k scores draft token x_{k+1}; row bs-1
 *                  scores the bonus position.
 *  draft_logits  : [B, bs-1, V]; row k is the drafter's score for x_{k+1}.
 *                  Unused (may be NULL) when temperature == 0.
 *  draft_tokens  : device int32 [B, bs-1]
 *  temperature   : > 0: p = softmax(l_t/T), q = softmax(l_d/T); accept x iff
 *                  u < min(1, p(x)/q(x)); at the first rejection emit the
 *                  inverse-CDF draw (vocabulary order) from max(0, p - q)
 *                  (from p if that mass is 0); if all bs-1 are accepted emit a
 *                  draw from p of row bs-1.  == 0: accept while x equals the
 *                  target argmax (lowest index on ties); emit the argmax at the
 *                  first mismatch, or of row bs-1.
 *  seed, cycle   : Philox-4x32-10 key (seed) and counter
 *                  (k, b, cycle_lo, cycle_hi); word 0 -> acceptance uniform,
 *                  word 1 -> draw uniform, uniform(w) = (w >> 8) * 2^-24.
 *  accepted_len  : device int32 [B], n in [0, bs-1]
 *  out_tokens    : device int32 [B, bs]: x_1 .. x_n, then the correction or
 *                  bonus token, then -1.
 * ------------------------------------------------------------------------- */
DFLASH_API size_t dflash_verify_workspace_size(int batch, int block_size, int vocab, dflash_dtype dtype);

DFLASH_API dflash_status dflash_verify(const void* target_logits, const void* draft_logits,
                            dflash_dtype dtype, const int32_t* draft_tokens,
                            int batch, int block_size, int vocab,
                            float temperature, uint64_t seed, uint64_t cycle,
                            int32_t* accepted_len, int32_t* out_tokens,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * 3b. Verification without a caller workspace.  The DFlash pages have no
 *     counterpart to this entry point; it serves callers that cannot allocate
 *     device memory when they verify -- code inside a CUDA graph being
 *     captured (cudaMalloc would break the capture), allocators that forbid
 *     late allocation, plain C hosts with no device allocator.
 *
 *  Same arguments and results as dflash_verify, minus the workspace.  Scratch
 *  comes from a static device array of dflash_verify_noalloc_max_scratch()
 *  bytes (4 MiB) that every GPU loading the library holds until exit; sizes
 *  needing more (dflash_verify_workspace_size() larger than that) are
 *  rejected with DFLASH_ERR_UNSUPPORTED and nothing is launched.  No call
 *  allocates or frees memory.  The first call on each device looks up the
 *  array's device address (cudaGetSymbolAddress) with that device current;
 *  make that first call before any stream capture.  All calls on a device
 *  share the array: calls that overlap on the GPU race, so order them on one
 *  stream.  The array keeps the last call's contents; nothing in it needs
 *  clearing because every entry is written before it is read.
 * ------------------------------------------------------------------------- */
DFLASH_API size_t dflash_verify_noalloc_max_scratch(void);

DFLASH_API dflash_status dflash_verify_noalloc(const void* target_logits, const void* draft_logits,
                                               dflash_dtype dtype, const int32_t* draft_tokens,
                                               int batch, int block_size, int vocab,
                                               float temperature, uint64_t seed, uint64_t cycle,
                                               int32_t* accepted_len, int32_t* out_tokens,
                                               void* stream);

/* ---------------------------------------------------------------------------
 * Diagnostics.
 * ------------------------------------------------------------------------- */

/* Test hook for the bounded waits inside the kernels (no counterpart in the
 * pages).  Runs only the last kernel of dflash_block_attn -- the one that
 * merges the key splits of each (sequence, KV head) once their writers have
 * counted in -- over counters that it clears and that nothing increments, with
 * its wait cut to limit_us microseconds (1..100000).  Every wait runs out:
 * the kernel raises DFLASH_DEV_TIMEOUT in the device status word, leaves `out`
 * untouched and returns, so the stream stays usable.  Arguments and workspace
 * as dflash_block_attn with window 0; bf16 caches only.  It reads the
 * sequence lengths and writes only the workspace's counters. */
DFLASH_API dflash_status dflash_debug_block_attn_wait_timeout(int batch, int block_size, int num_q_heads,
                                                             const dflash_kv_cache* cache, void* out,
                                                             void* workspace, size_t workspace_bytes,
                                                             unsigned limit_us, void* stream);

/* Philox-4x32-10 (Salmon et al., SC'11) on n device counters: ctr [n][4],
 * key [2] (host values), out [n][4].  The generator verification draws from. */
DFLASH_API dflash_status dflash_philox4x32_10(const uint32_t* ctr, uint32_t key0, uint32_t key1,
                                   uint32_t* out, int n, void* stream);

/* ---------------------------------------------------------------------------
 * 6. DFlash2 variants (DFlash & DFlash2 page, section 5).
 *
 * dflash_block_conv -- 5.1, the local depthwise 1D convolution along the
 *    block:  out_t = sum_{j=0}^{k-1} w_j (.) h_{t-j} + bias  (+ h_t if residual)
 *  h, out       : [batch * block_size, d_model] bf16, row b * block_size + t;
 *                 out may be h (in place).  Positions before a block's first
 *                 row contribute zero: the sum never crosses sequences.
 *  w            : [kernel, d_model] bf16 (per-channel taps, tap j on h_{t-j});
 *                 bias [d_model] bf16 or NULL.  kernel 1..8 (the pages use 3, 5).
 *  residual     : 1 adds h_t (the convolution as a sub-layer on the residual
 *                 stream between attention and the MLP), 0 the plain formula.
 *  Constraints: 1 <= block_size <= 16, d_model % 4 == 0, 8-byte aligned pointers.
 *
 * dflash_draft_topm -- 5.2, the candidate path selector's inputs: per draft
 *    position (row) of logits [batch, rows_per_seq, vocab] bf16, with
 *    P = softmax(logits / temperature), temperature > 0:
 *  idx_out      : [batch, rows_per_seq, m] int32, the m largest logits of the
 *                 row, larger first, ties to the lower index
 *  logp_out     : [batch, rows_per_seq, m] float, ln P of those candidates
 *  entropy_out  : [batch, rows_per_seq] float, -sum P ln P
 *  path_score_out: [batch] float, S = sum_j ln P(x_j^(m_j)) + lambda *
 *                 sum_j Entropy(P(x_j)) of the best path.  S is a sum of
 *                 per-position terms and the entropy term does not depend on
 *                 the choice, so the best path takes every position's first
 *                 candidate (a tree of candidates is idx_out itself).
 *  Constraints: 1 <= m <= 8, m <= vocab, 1 <= rows_per_seq <= 16,
 *               vocab % 8 == 0 and <= 524288, logits 16-byte aligned.
 * ------------------------------------------------------------------------- */
DFLASH_API dflash_status dflash_block_conv(const void* h, int batch, int block_size, int d_model, int kernel,
                                           const void* w, const void* bias, int residual, void* out, void* stream);

DFLASH_API size_t dflash_draft_topm_workspace_size(int batch, int rows_per_seq, int vocab, int m);

DFLASH_API dflash_status dflash_draft_topm(const void* logits, int batch, int rows_per_seq, int vocab, int m,
                                           float temperature, float lambda, int32_t* idx_out, float* logp_out,
                                           float* entropy_out, float* path_score_out, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * 5a. The start of a draft layer, before its attention (E4B page "The
 *    parameter count exposes the real cost": a Qwen3-style layer with q/k/v/o
 *    projections and two RMSNorms; "The released serving cycle": the drafter
 *    runs its layers over the block):
 *      h = RMSNorm(x) * g_in;  [q | k | v] = h W_qkv^T
 *
 *  x          : [batch * block_size, d_model] bf16 residual stream of the
 *               block rows (row b * block_size + j); only read
 *  g_in       : [d_model] the layer's input RMSNorm gain (NULL = ones)
 *  w_qkv      : [(num_q_heads + 2 * num_kv_heads) * 128, d_model] bf16: output
 *               rows h * 128 + e are query head h, then key heads, then value
 *               heads (element e of head g at row (num_q_heads + g) * 128 + e
 *               for keys, (num_q_heads + num_kv_heads + g) * 128 + e for values)
 *  q          : [batch, num_q_heads, block_size, 128] bf16 (dflash_block_attn's q)
 *  kb, vb     : [batch, num_kv_heads, block_size, 128] bf16 (its kb and vb)
 * The per-head Q/K RMSNorm and RoPE are dflash_block_attn's.  bf16 storage
 * points: the normalised rows and the three outputs.
 * Constraints: bf16; d_model % 128 == 0 and <= 4096; all pointers 16-byte
 *              aligned; workspace of dflash_draft_layer_qkv_workspace_size().
 * ------------------------------------------------------------------------- */
DFLASH_API size_t dflash_draft_layer_qkv_workspace_size(int batch, int block_size, int num_q_heads,
                                                       int num_kv_heads, int d_model);

DFLASH_API dflash_status dflash_draft_layer_qkv(const void* x, int batch, int block_size, int num_q_heads,
                                                int num_kv_heads, int d_model, const void* g_in, float eps,
                                                const void* w_qkv, void* q, void* kb, void* vb, void* workspace,
                                                size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * 5. The rest of a draft layer after its attention (E4B page "The parameter
 *    count exposes the real cost": a Qwen3-style layer, gated MLP of
 *    intermediate size 5120):
 *      x1 = x + o W_o^T;  h = RMSNorm(x1) * g_post;
 *      x2 = x1 + (silu(h W_gate^T) * (h W_up^T)) W_down^T
 *
 *  x          : [batch * block_size, d_model] bf16 residual stream of the
 *               block rows (row b * block_size + j); overwritten with x2
 *  attn_out   : [batch, num_q_heads, block_size, 128] bf16 (dflash_block_attn's out)
 *  w_o        : [d_model, num_q_heads * 128]
 *  g_post     : [d_model] post-attention RMSNorm gain (NULL = ones)
 *  w_gate_up  : [2 * mlp_dim, d_model], gate and up rows interleaved in blocks of
 *               64: rows 128t .. 128t+63 = gate rows 64t .. 64t+63, rows
 *               128t+64 .. 128t+127 = up rows 64t .. 64t+63
 *  w_down     : [d_model, mlp_dim]
 * bf16 storage points: x1, the normalised rows, the SwiGLU activations, x2.
 * Constraints: bf16; d_model % 128 == 0 and <= 4096; mlp_dim % 64 == 0;
 *              128 % block_size == 0; all pointers 16-byte aligned.
 * ------------------------------------------------------------------------- */
DFLASH_API size_t dflash_draft_layer_tail_workspace_size(int batch, int block_size, int num_q_heads, int d_model,
                                              int mlp_dim);

DFLASH_API dflash_status dflash_draft_layer_tail(void* x, const void* attn_out, int batch, int block_size,
                                      int num_q_heads, int d_model, int mlp_dim, const void* w_o,
                                      const void* g_post, const void* w_gate_up, const void* w_down, float eps,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * 4. The drafter's head: final RMSNorm, LM head and draft sampling.
 *    E4B page "The released serving cycle" (the drafter proposes the block's
 *    tokens from its final hidden states through its LM head) and "The
 *    parameter count exposes the real cost" (the V x D head).
 *
 *  x            : [batch * rows_per_seq, d_model] bf16 final hidden states of
 *                 the proposal rows, row b * rows_per_seq + k = sequence b,
 *                 proposal k (the block's rows 1 .. bs-1: rows_per_seq = bs-1)
 *  g_final      : [d_model] final RMSNorm gain (NULL = ones); eps its epsilon
 *  w_head       : [vocab, d_model] bf16, row v = token v
 *  temperature  : > 0: token = argmax_y logits[y]/T - ln(-ln U_y), a draw from
 *                 softmax(logits/T) (the exponential race); U_y from
 *                 Philox-4x32-10 with key (seed_lo, seed_hi) and counter
 *                 (y >> 2, (b << 5) | k, cycle_lo, cycle_hi | 2^31), word y & 3,
 *                 U = ((w >> 8) + 1) * 2^-24 (cycle < 2^63).  == 0: argmax.
 *                 Ties go to the lowest index.
 *  logits_out   : [batch * rows_per_seq, vocab] bf16 (the draft logits that
 *                 dflash_verify takes)
 *  tokens_out   : device int32 [batch * rows_per_seq], the draft tokens
 * Constraints: bf16 only; d_model % 64 == 0; vocab % 128 == 0;
 *              1 <= rows_per_seq <= 31; x, w_head, logits 16-byte aligned.
 * ------------------------------------------------------------------------- */
DFLASH_API size_t dflash_draft_head_workspace_size(int batch, int rows_per_seq, int d_model, int vocab);

DFLASH_API dflash_status dflash_draft_head(const void* x, int batch, int rows_per_seq, int d_model,
                                const void* g_final, float eps, const void* w_head, int vocab,
                                float temperature, uint64_t seed, uint64_t cycle,
                                void* logits_out, int32_t* tokens_out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, returns the device status word (DFLASH_DEV_* bits)
 * in *flags and clears it on the current device. */
DFLASH_API dflash_status dflash_read_device_status(uint32_t* flags, void* stream);

/* Text of the last host-side error of the calling thread ("" if none). */
DFLASH_API const char* dflash_last_error_string(void);

/* ABI version: (major << 16) | minor. */
DFLASH_API int dflash_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H_ */
