/*
 * gbattn.h - C ABI of the GB300 (sm_103a) fused attention library.
 *
 * The operation.  Multi-head attention O = softmax(Q K^T * scale, mask) V with
 * the row log-sum-exp LSE, computed block by block with a running max/sum
 * correction so that the [batch, head, seq, seq] score matrix never reaches
 * device memory (smzdm contest article "杀进决赛!这 28 支队伍把算子优化卷疯了!",
 * section 03, on how FlashAttention tiles and fuses standard attention;
 * zwxr.cn CANN ops-nn fused-attention article, sections 3.1-3.3, for the
 * operator's inputs, mask and key-block loop with online softmax), and its
 * backward pass dQ, dK, dV from the recomputed attention matrix (smzdm article,
 * section 03, on the three gradients of the contest's Sparse FlashAttention
 * backward operator), with an optional block-sparse mask whose skipped tiles are
 * never computed (same section, on sparsity).
 *
 * Definitions (all positions relative to the start of their sequence):
 *   keep(i, j)  = j < L  and  [none: true | causal: j <= i |
 *                 block: tile (i/64, j/64) listed and (causal_in_block ? j <= i : true)]
 *   s_ij        = scale * <q_i, k_j>             (masked: -inf)
 *   LSE_i       = ln sum_j exp(s_ij)              (natural log, float32)
 *   O_i         = sum_j exp(s_ij - LSE_i) v_j
 *   dP_ij       = <dO_i, v_j>;  D_i = <dO_i, O_i>;  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i = scale sum_j dS_ij k_j;  dK_j = scale sum_{h in group} sum_i dS_ij q_i;
 *   dV_j = sum_{h in group} sum_i P_ij dO_i
 * A row with no allowed key gets O = 0 and LSE = -inf and adds nothing to any
 * gradient.  Query head h reads KV head h / (heads_q / heads_kv).
 *
 * Memory and ownership.  Every pointer argument is caller-owned device memory
 * unless marked "host".  The library never allocates or frees device memory:
 * scratch space is the caller's `workspace` of at least the size the matching
 * *_workspace_size() call returns.  The library itself holds one device status
 * word per GPU and nothing else.
 *
 * Layouts.  Elements are float32 (ATTN_F32) or bfloat16 (ATTN_BF16); the head
 * dimension is always contiguous.
 *   fixed length    q, o, dout, dq: [batch, heads_q, seqlen, head_dim] by strides
 *                   q_stride_b/h/s (in elements); k, v, dk, dv: [batch, heads_kv,
 *                   seqlen, head_dim] by kv_stride_b/h/s.  lse: contiguous float32
 *                   [batch, heads_q, seqlen].
 *   variable length (cu_seqlens != NULL) tokens of all sequences packed:
 *                   q-like [T, heads_q, head_dim], kv-like [T, heads_kv, head_dim],
 *                   row of position s of sequence n = cu_seqlens[n] + s, strides
 *                   *_stride_s (between tokens) and *_stride_h; *_stride_b ignored.
 *                   lse: contiguous float32 [heads_q, T].
 *
 * Constraints.  head_dim 64, 128 or 256 (both types; bf16 runs on the tensor
 * cores at every head dim, the deterministic backward at 64 and 128 only);
 * heads_q % heads_kv == 0; every tensor pointer 16-byte aligned; strides
 * multiples of 8 elements (16 bytes) for bf16 and 4 elements for float32.
 *
 * Errors.  Every argument error is detected on the host and returned before any
 * device work is queued; outputs are then left untouched.  Errors found on the
 * device are recorded in the device status word and returned by
 * attn_get_status(): a bounded pipeline wait that ran out
 * (ATTN_ERR_DEVICE_TIMEOUT), and, in the checked build of this library
 * (libgbattn_checked.so, compiled with GBATTN_CHECKED=1; attn_version() ends in
 * " checked"), an index computed on the device that lies outside its tensor
 * (ATTN_ERR_DEVICE_BOUNDS).  The checked build compares every work-list entry,
 * block-mask entry read on the device, and the sequence, head and position
 * behind each tile load, reduce-add, row read and row store of the attention
 * kernels with the tensor's extent before the access, and skips the access if
 * the check fails.  With valid arguments no check fails; the plain build
 * carries no checks.
 *
 * Asynchrony.  attn_fwd and attn_bwd only queue work on `stream` (a cudaStream_t;
 * NULL = the legacy default stream) and return; outputs are ready once the
 * stream reaches that point.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* a shape, stride, pointer or index list is invalid */
  ATTN_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. head_dim 96) */
  ATTN_ERR_WORKSPACE = 3,      /* workspace NULL, misaligned or smaller than required */
  ATTN_ERR_CUDA = 4,           /* a CUDA runtime call failed (no device, launch error) */
  ATTN_ERR_DEVICE_TIMEOUT = 5, /* device: a bounded pipeline wait gave up */
  ATTN_ERR_DEVICE_BOUNDS = 6   /* device: an index check failed; the access was skipped */
} attn_status_t;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype_t;

typedef enum { ATTN_MASK_NONE = 0, ATTN_MASK_CAUSAL = 1, ATTN_MASK_BLOCK = 2 } attn_mask_t;

/*
 * Block-sparse mask: which 64x64 tiles of the [seq, seq] score matrix are computed
 * (smzdm article, section 03: tiles that need no computation are skipped).  CSR by
 * query row block; column indices strictly ascending inside a row.  One mask serves
 * every batch entry and head.  Both copies must hold the same lists: the host copy
 * is validated, the device copy is read by the kernels.
 */
typedef struct {
  const int32_t* row_ptr;      /* device, [n_row_blocks + 1], row_ptr[0] = 0 */
  const int32_t* col_idx;      /* device, [nnz] */
  const int32_t* row_ptr_host; /* host copy of row_ptr */
  const int32_t* col_idx_host; /* host copy of col_idx */
  int32_t block_q, block_k;    /* tile size: must be 64 and 64 */
  int32_t n_row_blocks;        /* = ceil(seqlen / 64) */
  int32_t n_col_blocks;        /* = ceil(seqlen / 64) */
  int32_t nnz;                 /* = row_ptr[n_row_blocks] */
  int32_t causal_in_block;     /* 1: inside listed tiles also require j <= i */
} attn_block_mask_t;

typedef struct {
  int32_t batch;        /* fixed length: batch size (variable length: ignored) */
  int32_t heads_q;      /* query heads Hq */
  int32_t heads_kv;     /* key/value heads Hkv, Hq % Hkv == 0 (GQA when Hkv < Hq) */
  int32_t seqlen;       /* fixed length: S; variable length: >= the longest sequence */
  int32_t head_dim;     /* D */
  const int32_t* cu_seqlens;      /* device [n_seqs + 1] sequence starts, or NULL */
  const int32_t* cu_seqlens_host; /* host copy, required when cu_seqlens != NULL */
  int32_t n_seqs;                 /* number of packed sequences */
  int64_t q_stride_b, q_stride_h, q_stride_s;    /* q, o, dout, dq (elements) */
  int64_t kv_stride_b, kv_stride_h, kv_stride_s; /* k, v, dk, dv (elements) */
  float scale;          /* score scale, usually 1/sqrt(D) */
  attn_dtype_t dtype;   /* element type of q, k, v, o, dout, dq, dk, dv */
  attn_mask_t mask;
  const attn_block_mask_t* block_mask; /* host struct; required iff mask == ATTN_MASK_BLOCK */
} attn_params_t;

/*
 * Bytes of device workspace attn_fwd / attn_bwd need for these parameters, or
 * SIZE_MAX if the parameters are invalid (attn_last_error() says why).  The
 * backward workspace holds the float32 dQ accumulator [rows, heads_q, D], the
 * per-row D_i = <dO_i, O_i>, the work list and, for block masks, the transposed
 * (per key block) tile lists.  The forward workspace holds the work list and,
 * when there are few work units for long sequences (each unit's key range is
 * then split into parts run on separate SMs), the parts' float32 partial results.
 * With fewer units than a GB300 has SMs the bf16 forward lists one 128-row query
 * tile per unit instead of two, which doubles its work list; the size returned
 * covers both that list and the FP8 forward's, so one query serves attn_fwd and
 * attn_fwd_fp8.
 */
size_t attn_fwd_workspace_size(const attn_params_t* p);
size_t attn_bwd_workspace_size(const attn_params_t* p);

/*
 * Forward: O and LSE for the definitions above (zwxr.cn CANN ops-nn article,
 * section 3.3: per query block, stream key/value blocks, scale the dot products,
 * mask to -inf, keep the running max and sum, accumulate exp(score - max) V).
 * q, k, v: inputs; o: output (same layout as q); lse: float32 output;
 * workspace: caller-owned device scratch, 256-byte aligned, >= attn_fwd_workspace_size.
 * Returns ATTN_OK once the work is queued, or an error before queuing anything.
 */
attn_status_t attn_fwd(const attn_params_t* p, const void* q, const void* k, const void* v,
                       void* o, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * Backward: dQ, dK, dV from q, k, v, the forward's o and lse, and dout = dL/dO
 * (smzdm article, section 03: the attention matrix is recomputed block by block,
 * two gradients gather along the key direction and the third is accumulated by
 * many blocks into the same place).  dk and dv are sums over the query heads of
 * each KV head's group.  dq, dk, dv: outputs with the q / kv layouts; workspace
 * as for attn_fwd with attn_bwd_workspace_size bytes.  dQ is accumulated in
 * float32 by L2 reductions whose order is not fixed, so its last bits may
 * differ from run to run (see attn_bwd_deterministic).
 */
attn_status_t attn_bwd(const attn_params_t* p, const void* q, const void* k, const void* v,
                       const void* o, const void* dout, const float* lse, void* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Deterministic backward: the same outputs as attn_bwd, bit-identical from run
 * to run.  The pages point at both causes and the cure: the dQ sum's order
 * varies with the order in which blocks add into it (zwxr.cn CANN article,
 * section 6.1), and the backward can walk the blocks in the other loop order
 * (smzdm contest article, section 03).  Here dK and dV come from the
 * dK/dV-stationary pass without its dQ product, and dQ from a second,
 * query-stationary pass that recomputes S and dP per query tile and sums over
 * key tiles in ascending order (three products per tile instead of one, so
 * the backward does 7 products instead of 5).  Arguments, layouts and the
 * workspace (attn_bwd_workspace_size bytes) are those of attn_bwd.  Only the
 * tensor-core path (bf16, head_dim 64 or 128) has it: float32 and head_dim
 * 256 return ATTN_ERR_UNSUPPORTED before queuing anything.
 */
attn_status_t attn_bwd_deterministic(const attn_params_t* p, const void* q, const void* k, const void* v,
                                     const void* o, const void* dout, const float* lse, void* dq, void* dk,
                                     void* dv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 (e4m3) forward.  Newer accelerators multiply 8-bit floats so that each
 * transfer and each matrix instruction handles more numbers, while sums are
 * kept in a wider format so that small terms are not lost (smzdm contest
 * article, closing section on precision).  The pages fix no format or scaling;
 * this library's choices:
 *
 * Format: E4M3 of the OCP 8-bit floating-point specification without
 * infinities (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest
 * finite value 448, smallest subnormal 2^-9).
 *
 * attn_quantize_fp8: for each 128-row tile (positions r0 .. r0 + 127, the last
 * one possibly short) of each head of q, k and v (bf16, laid out and strided
 * as for attn_fwd), amax = max |x| over the tile; scale = amax / 448 and
 * code = e4m3(x * (448 / amax)), the division and the product rounded to
 * float32, the conversion rounded to nearest even and saturated at +-448; an
 * all-zero tile gets scale 0 and zero codes.  A code stands for
 * e4m3_value(code) * scale.  Outputs (contiguous, caller-owned device memory):
 *   q8  [batch, heads_q, seqlen, 128] bytes;  k8 [batch, heads_kv, seqlen, 128] bytes;
 *   v8t [batch, heads_kv, 128, ld] bytes with ld = seqlen rounded up to 16: V's
 *       codes transposed, keys along each row (positions seqlen .. ld-1 unwritten);
 *   q_scale [batch, heads_q, n_tiles], k_scale and v_scale [batch, heads_kv, n_tiles]
 *       float32, n_tiles = ceil(seqlen / 128).
 * Device-memory bound: 2 bytes read and 1 written per element.
 *
 * attn_fwd_fp8: O and LSE of attention on the dequantised q, k, v (the
 * definitions at the top of this file, every mask kind, GQA) with both products
 * on e4m3 operands and float32 accumulation.  The Q and K tile scales fold into
 * the score scale; each V tile's scale, relative to the largest V tile scale of
 * its KV head, folds into P, which is rounded to e4m3 before the P V product
 * (that rounding is the one approximation beyond float32 rounding: it moves
 * each output element by at most sum_j (2^-4 P_ij + min(P_ij, 2^-10 / (l_i r_j)))
 * |v_jd|, with l_i the row's sum of exp(s_ij - max_j s_ij) and r_j the V scale
 * ratio).  LSE is computed from the unrounded P.  o: bf16, laid out by the q
 * strides as for attn_fwd; lse: float32 [batch, heads_q, seqlen]; workspace:
 * attn_fwd_workspace_size(p) bytes.
 *
 * Both calls: p->dtype must be ATTN_BF16, p->head_dim 128 and p->cu_seqlens NULL
 * (else ATTN_ERR_UNSUPPORTED); byte tensors 16-byte aligned, scale arrays 4-byte
 * aligned; inputs must be finite.  p's q strides give the bf16 q (quantisation)
 * and o (forward); its kv strides give the bf16 k and v of the quantisation and
 * are validated by the forward like attn_fwd's (the codes' own layouts above are
 * fixed).  Errors and asynchrony as for attn_fwd.
 */
attn_status_t attn_quantize_fp8(const attn_params_t* p, const void* q, const void* k, const void* v, void* q8,
                                void* k8, void* v8t, float* q_scale, float* k_scale, float* v_scale, void* stream);
attn_status_t attn_fwd_fp8(const attn_params_t* p, const void* q8, const void* k8, const void* v8t,
                           const float* q_scale, const float* k_scale, const float* v_scale, void* o, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass that allocates nothing.  The pages have no counterpart to this
 * entry point: it exists for callers that may not allocate device memory and so
 * cannot pass a workspace -- engines that fix their device memory budget at
 * start-up and forbid any later allocation, and plug-ins inside a host
 * framework that owns the device allocator and shares none of it.
 *
 * Same arguments, results and errors as attn_bwd, minus the workspace: scratch
 * space is a fixed array of ATTN_NOALLOC_SCRATCH_BYTES inside the library's device
 * memory, which every GPU that loads the library holds until the process exits.
 * A problem whose attn_bwd_workspace_size() exceeds that size is rejected with
 * ATTN_ERR_WORKSPACE before anything is queued (attn_last_error() gives both
 * sizes), after the argument checks attn_bwd makes, so an invalid argument gets
 * attn_bwd's code.  The first call on each device looks up the array's device
 * address (with that device current); make that first call before any stream
 * capture.  Every call shares the one array: calls whose work overlaps on the
 * GPU race on it, so queue them on one stream or wait between them.  No call
 * depends on what a previous call left in the array.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
attn_status_t attn_bwd_noalloc(const attn_params_t* p, const void* q, const void* k, const void* v,
                               const void* o, const void* dout, const float* lse, void* dq, void* dk,
                               void* dv, void* stream);

/*
 * Waits for `stream`, then returns and clears the device status word of the
 * current device (ATTN_OK if no device-side error was recorded).
 */
attn_status_t attn_get_status(void* stream);

/* Static string naming a status code. */
const char* attn_status_string(attn_status_t s);

/* Thread-local text describing the last argument error of this thread ("" if none). */
const char* attn_last_error(void);

/*
 * Measurement hook.  While set, every attn_fwd (which = 0) or attn_bwd (which = 1)
 * made by the calling thread records the CUDA event `start` on its stream just
 * before launching its main attention kernel(s) and `stop` just after, so a
 * caller can time them alone; which = 2 and 3 bracket the backward's
 * preprocess (D and the accumulator zero-fill) and its dQ conversion.  `start`
 * and `stop` are cudaEvent_t handles owned by the caller; NULL clears the hook.
 * Returns ATTN_ERR_INVALID_ARG for an unknown `which`.
 */
attn_status_t attn_set_timing_events(int which, void* start, void* stop);

/* Library version, e.g. "gbattn 0.1.0 sm_103a". */
const char* attn_version(void);

/*
 * Self-test of the device-side timeout path (the pages have no counterpart:
 * it checks this library's own failure handling).  Queues one small kernel in
 * which a warp waits, through the same bounded mbarrier wait every
 * tensor-core kernel uses, on a barrier that nothing completes.  After
 * limit_us microseconds (1 .. 1000000) the wait gives up, records
 * ATTN_ERR_DEVICE_TIMEOUT in the device status word and the kernel returns:
 * nothing faults, traps or hangs, and the context stays usable.  The next
 * attn_get_status() on the stream returns ATTN_ERR_DEVICE_TIMEOUT (and clears
 * it).  Returns ATTN_OK once queued, ATTN_ERR_INVALID_ARG for a limit out of
 * range.
 */
attn_status_t attn_selftest_bounded_wait(unsigned int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
