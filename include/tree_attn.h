/*
 * tree_attn.h -- C ABI of the tree-packed training hot path (GB300 / sm_103a).
 *
 * Tree packing stores every token of a set of sequences that share prefixes
 * once, in depth-first (preorder) order, so that one forward/backward pass
 * computes each shared prefix a single time:
 *   - Tree Training: Accelerating Agentic LLMs Training via Shared Prefix Reuse
 *     (arXiv 2511.00413), cited below as [TT];
 *   - Trie packing, agillm.io visualisation, cited as [TP];
 *   - Claw-R1 documentation "Prefix Tree Merge", cited as [PTM].
 *
 * Conventions shared by every call
 *   - Row i of a packed tree is the token at preorder index i; its preorder
 *     index IS i, so no separate preorder array exists.
 *   - The ancestor mask is never stored densely. Key j is visible to query i
 *     iff  j <= i <= subtree_end[j]  (subtree_end[j] = last row of j's
 *     subtree). This per-key interval form equals [TT] §3.2 "Attention Mask"
 *     (j <= i and both on one root-to-leaf path) and [TT] Appendix A.1
 *     (whole ancestor chunks, causal inside a token's own chunk).
 *   - Tensors are dense, row-major, contiguous, with no padding:
 *       Q, dQ, O, dO [T, Hq, d];  K, V, dK, dV [T, Hkv, d];  LSE [Hq, T] fp32;
 *       hidden, d_hidden [T, K_h];  W_LM, dW [K_h, V].
 *     Query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups).
 *   - dtype is TREE_DTYPE_BF16 (bf16 storage, fp32 accumulation on tensor
 *     cores) or TREE_DTYPE_F32 (fp32 storage and arithmetic).
 *   - Pointers named "device" are CUDA device addresses owned by the caller;
 *     the library never allocates or frees device memory. Scratch space is the
 *     caller's `workspace` (device, at least the size returned by the matching
 *     *_workspace_size query, 256-byte aligned), with one exception:
 *     tree_attn_fwd_noalloc keeps its scratch in a fixed device array that the
 *     library holds (see that entry).
 *   - Every device call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and returns after enqueueing its kernels.
 *   - Every call returns a tree_status. Argument errors are found on the host
 *     before anything is enqueued and leave outputs untouched. Device-side
 *     range checks never trap: they set a device error word that
 *     tree_check_device_status() reads. tree_last_error() describes the most
 *     recent failure on the calling host thread. No C++ exception crosses
 *     this interface.
 */
#ifndef TREE_ATTN_H_
#define TREE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* tree_stream_t;

typedef enum {
  TREE_OK = 0,
  TREE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad flag */
  TREE_ERR_SHAPE = 2,         /* unsupported or inconsistent sizes */
  TREE_ERR_DTYPE = 3,         /* dtype not one of TREE_DTYPE_* */
  TREE_ERR_ALIGNMENT = 4,     /* pointer not 16-byte (workspace: 256-byte) aligned */
  TREE_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
  TREE_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up */
  TREE_ERR_DEVICE_CHECK = 7,  /* a device-side range check failed */
  TREE_ERR_WORKSPACE = 8      /* workspace smaller than the size query says */
} tree_status;

typedef enum { TREE_DTYPE_F32 = 0, TREE_DTYPE_BF16 = 1 } tree_dtype;

/* ------------------------------------------------------------------------ */
/* Host packing                                                              */
/* ------------------------------------------------------------------------ */
/*
 * Packing follows [TP] "Step 1 - Store each node once" (a token is shared
 * only when its whole preceding context is identical; position = depth),
 * [TT] §3.1 eq. 8 (DFS serialisation), [TT] §3.2 eq. 9 (positions) and
 * [PTM] "1. build and compress" (insert into a trie, compress single-child
 * chains into nodes, number nodes in preorder).
 *
 * Readings fixed by this interface:
 *   - children and roots are ordered by first insertion (both worked examples);
 *   - several distinct first tokens give a forest; positions restart at 0;
 *   - a node (chunk) ends at a fork, at a leaf, and where an input sequence
 *     ends ([PTM]'s node list);
 *   - occurrences are the original next-token predictions ([TP] "Share
 *     logits, preserve every prediction"): for each input sequence k in input
 *     order and t = 0 .. len_k - 2, (row of token t, token t+1, weight w_k);
 *     duplicated sequences keep their own occurrences; no EOS is added.
 *
 * Two phases so that the caller owns every output array:
 *   tree_pack_plan() builds the trie and reports sizes; the caller allocates;
 *   tree_pack_emit() fills the arrays; tree_plan_free() releases the plan.
 */
typedef struct tree_plan tree_plan;

typedef struct {
  int64_t T;          /* packed rows (unique prefixes) */
  int64_t n_nodes;    /* compressed nodes (chunks) */
  int64_t n_occ;      /* next-token occurrences = sum_k max(len_k - 1, 0) */
  int64_t n_roots;    /* trees in the forest */
  int64_t n_tokens;   /* total input tokens = seq_offsets[n_seqs] */
} tree_pack_sizes;

/* Host arrays, caller-allocated; any pointer may be NULL to skip that output. */
typedef struct {
  int32_t* packed_ids;      /* [T]   token id of row i */
  int32_t* position_ids;    /* [T]   depth of row i (eq. 9) */
  int32_t* subtree_end;     /* [T]   last row of row i's subtree (>= i) */
  int32_t* path_count;      /* [T]   input sequences whose path holds row i */
  int32_t* parent_row;      /* [T]   parent row, -1 for a root */
  int32_t* node_of_token;   /* [T]   node (chunk) holding row i */
  int32_t* node_start;      /* [n_nodes] first row of the node */
  int32_t* node_end;        /* [n_nodes] last row of the node (inclusive) */
  int32_t* node_parent;     /* [n_nodes] parent node, -1 for a root node */
  int32_t* token_rows;      /* [n_tokens] packed row of every input token (unpacking map) */
  int32_t* occ_source_rows; /* [n_occ] row whose logits make the prediction */
  int32_t* occ_targets;     /* [n_occ] predicted token id */
  int32_t* occ_seq;         /* [n_occ] input sequence of the occurrence */
  float*   occ_weights;     /* [n_occ] weight of that sequence (1.0 if none given) */
  int32_t* occ_row_ptr;     /* [T+1] CSR: occurrences of row r are
                                occ_perm[occ_row_ptr[r] .. occ_row_ptr[r+1]) */
  int32_t* occ_perm;        /* [n_occ] occurrence ids stably sorted by source row */
} tree_pack_out;

/* tokens: host [n_tokens] int32; seq_offsets: host [n_seqs+1] int64, nondecreasing,
 * seq_offsets[0] == 0. Writes a new plan to *plan (free with tree_plan_free) and
 * its sizes to *sizes. Errors: TREE_ERR_INVALID_ARG (null pointers, bad offsets),
 * TREE_ERR_SHAPE (more than 2^31 - 1 rows or occurrences). */
int tree_pack_plan(const int32_t* tokens, const int64_t* seq_offsets, int64_t n_seqs,
                   tree_plan** plan, tree_pack_sizes* sizes);

/* seq_weights: host [n_seqs] or NULL (all 1.0). Fills the non-NULL arrays of *out. */
int tree_pack_emit(const tree_plan* plan, const float* seq_weights, const tree_pack_out* out);

void tree_plan_free(tree_plan* plan);

/* Host check that subtree_end (host [T]) is a preorder forest: i <= end[i] < T and
 * the intervals [i, end[i]] nest. TREE_OK or TREE_ERR_INVALID_ARG. */
int tree_validate_subtree_end(const int32_t* subtree_end, int64_t T);

/* ------------------------------------------------------------------------ */
/* RoPE on depth positions                                                   */
/* ------------------------------------------------------------------------ */
/*
 * [TT] §3.2 "Position Embedding" (eq. 9) and [TP] Step 1: every row is rotated
 * by its depth position, so packed rows see the rotation of their own
 * per-path sequence. Variant (the pages name RoPE only): rotate-half pairs
 * (x[k], x[k + d/2]) turned by angle pos * theta_base^(-2k/d), k < d/2; the
 * angle is formed in fp32 and sin/cos are CUDA's accurate sincosf.
 * inverse = 1 applies the transposed rotation (the backward of the forward
 * rotation, used on dQ/dK).
 *
 * q: device [T, Hq, d], k: device [T, Hkv, d], rotated in place (either may be
 * NULL); position_ids: device [T] int32, >= 0. d even, 2 <= d <= 256.
 */
int tree_rope(void* q, void* k, const int32_t* position_ids, int64_t T, int Hq, int Hkv,
              int d, float theta_base, int dtype, int inverse, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Tree attention                                                            */
/* ------------------------------------------------------------------------ */
/*
 * Forward ([TP] "Step 2 - Allow only ancestors and self", "Step 3";
 * [TT] §3.2 "Attention Mask", eq. 6 forward equivalence):
 *   O_i   = sum_{j : j <= i <= subtree_end[j]} softmax_j(q_i . k_j * scale) v_j
 *   LSE_i = ln sum_{same j} exp(q_i . k_j * scale)          (per query head)
 * scale = softmax_scale if > 0, else 1/sqrt(d). No dropout, no softcap.
 *
 * Backward ([TP] "Same chain rule, shared computation graph", Step 3: a key
 * collects the gradients of every descendant query that sees it):
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - Delta_i),
 *   Delta_i = dO_i . O_i,  dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 * with dK/dV of a KV head summed over its query heads.
 *
 * Sizes: 1 <= T < 2^31, Hq % Hkv == 0, d in {64, 128}. q, k, v, o, dout, dq, dk,
 * dv: device, 16-byte aligned, dtype elements; lse: device fp32 [Hq, T];
 * subtree_end: device int32 [T]. Rows with an out-of-range subtree_end
 * (end < i or end >= T) set TREE_ERR_DEVICE_CHECK in the device error word;
 * outputs are then unspecified (never out-of-bounds accesses). Nesting is not
 * checked on the device (see tree_validate_subtree_end).
 * deterministic: 0 lets dQ, dK and dV accumulate with fp32 reductions from work units
 * that run in any order (results may differ in the last bits run to run); 1 makes
 * every sum fixed-order and the results bitwise reproducible: dK and dV come from one
 * work unit per key tile, and dQ from a second, query-stationary pass that walks each
 * query tile's key tiles in order (S and dP recomputed: more FLOPs, slower). The
 * kernels at head size 64 (below) always sum in one fixed order, so there both values
 * give bitwise reproducible results.
 *
 * Kernels by (dtype, d) -- tree_kernel_path tells which a call takes:
 *   bf16, d = 128   tcgen05 kind::f16 (bf16 operands, fp32 TMEM accumulators), TMA-fed.
 *   fp32 or bf16, d = 64   tcgen05 kind::tf32 with every fp32 operand split into
 *                   hi = tf32(x) and lo = tf32(x - hi), products taken as hi.hi + hi.lo
 *                   + lo.hi (about 2^-21 relative error each; terms with an exactly
 *                   representable operand are skipped).
 *   fp32, d = 128   CUDA cores (fp32 FMA): the hi/lo tiles of a 128-row, 128-wide fp32
 *                   operand pair do not fit a CTA's shared memory next to each other.
 */
size_t tree_attn_workspace_size(int64_t T, int Hq, int Hkv, int d, int dtype);

int tree_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int32_t* subtree_end, int64_t T, int Hq, int Hkv, int d, int dtype,
                  float softmax_scale, void* workspace, size_t workspace_bytes,
                  tree_stream_t stream);

/*
 * tree_attn_fwd_noalloc -- the same forward as tree_attn_fwd, for callers that
 * cannot allocate device memory for a workspace (a framework whose pool already
 * owns the device memory it may use, a serving loop that forbids cudaMalloc after
 * start-up, a plugin interface with no workspace slot). The pages have no
 * counterpart to this call; it only changes where the scratch lives.
 *
 * Its scratch is a fixed ~276 KB array in device memory inside the library, held
 * on every GPU that loads the library until the process exits. T may not exceed
 * 65536 rows (TREE_ERR_SHAPE otherwise); the other arguments and the results are
 * those of tree_attn_fwd. All calls share the array: calls whose kernels overlap
 * on the GPU (e.g. on two streams) race, so keep them ordered on one stream. Each
 * call rewrites every scratch entry it reads. The first call on a device looks up
 * the array's device address, so make it before any stream capture. No call
 * allocates or frees device memory.
 */
int tree_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* subtree_end, int64_t T, int Hq, int Hkv, int d,
                          int dtype, float softmax_scale, tree_stream_t stream);

int tree_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv,
                  const int32_t* subtree_end, int64_t T, int Hq, int Hkv, int d, int dtype,
                  float softmax_scale, int deterministic, void* workspace,
                  size_t workspace_bytes, tree_stream_t stream);

/*
 * tree_attn_bwd_rope -- tree_attn_bwd, then the backward of the depth rotation
 * (tree_rope with inverse = 1) on dq and dk, in one pass: when q = R q0 and
 * k = R k0 came from tree_rope, it returns dL/dq0 = R^T dL/dq and dL/dk0 =
 * R^T dL/dk (dv unchanged). On the tensor-core path the rotation is applied to
 * the fp32 sums before their one rounding to dtype, inside the kernel that
 * writes dq and dk; elsewhere it is a tree_rope call after the backward.
 * Arguments as tree_attn_bwd, plus position_ids (device int32 [T], >= 0) and
 * theta_base (finite, > 1) as in tree_rope.
 */
int tree_attn_bwd_rope(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       const int32_t* subtree_end, const int32_t* position_ids, int64_t T,
                       int Hq, int Hkv, int d, int dtype, float softmax_scale,
                       float theta_base, int deterministic, void* workspace,
                       size_t workspace_bytes, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Shared-logit log-probs                                                    */
/* ------------------------------------------------------------------------ */
/*
 * Forward ([TP] "Share logits, preserve every prediction" and "The
 * training-loop change is small"): z_r = hidden_r W_LM (never stored),
 *   lse[r]  = ln sum_v exp(z_rv)                  for every row r in [0, T)
 *   logp[o] = z_{r_o, y_o} - lse[r_o]             for every occurrence o
 * with r_o = source row, y_o = occ_targets[o]. Occurrences are reached through
 * the row CSR (occ_row_ptr [T+1], occ_perm [n_occ]) from tree_pack_emit.
 *
 * Backward ([TP] "Same chain rule, shared computation graph", Step 1;
 * [TT] §3.2 "Loss Weights"): with g_o = grad_logp[o] = dL/dlogp_o
 * (= -w_o for the weighted loss L = -sum_o w_o logp_o),
 *   G_z[r]   = sum_{o at r} g_o (e_{y_o} - softmax(z_r))   (targets at a shared row add)
 *   d_hidden = G_z W_LM^T,   d_w = hidden^T G_z            (both overwritten)
 * z is recomputed from hidden, W_LM and lse.
 *
 * hidden, d_hidden: device [T, K_h]; w_lm, d_w: device [K_h, V]; dtype elements,
 * 16-byte aligned; K_h % 64 == 0 and V % 8 == 0. lse: device fp32 [T];
 * logp, grad_logp: device fp32 [n_occ]; index arrays device int32.
 * Out-of-range targets or CSR entries set TREE_ERR_DEVICE_CHECK and are skipped.
 *
 * Kernels: bf16 runs the tcgen05 kind::f16 GEMM with the LSE / G_z / dW-correction
 * epilogues; fp32 runs tcgen05 kind::tf32 GEMMs with the two-term operand split
 * (hi.hi + hi.lo + lo.hi) and the same epilogue arithmetic, G_z kept in fp32.
 */
size_t tree_logprob_workspace_size(int64_t T, int64_t K_h, int64_t V, int64_t n_occ, int dtype);

int tree_logprob_fwd(const void* hidden, const void* w_lm, const int32_t* occ_row_ptr,
                     const int32_t* occ_perm, const int32_t* occ_targets, int64_t T,
                     int64_t K_h, int64_t V, int64_t n_occ, float* lse, float* logp,
                     int dtype, void* workspace, size_t workspace_bytes,
                     tree_stream_t stream);

/* dw_fp32 = 1 writes d_w in fp32 ([K_h, V] floats: the fp32 accumulation itself, for a
 * caller that keeps fp32 master weights; [TT] Appendix B.5 keeps gradients summed over
 * shared rows in fp32), 0 writes it in dtype. With TREE_DTYPE_F32 d_w is fp32 either way.
 * Any other value: TREE_ERR_INVALID_ARG. */
int tree_logprob_bwd(const void* hidden, const void* w_lm, const float* lse,
                     const int32_t* occ_row_ptr, const int32_t* occ_perm,
                     const int32_t* occ_targets, const float* grad_logp, int64_t T,
                     int64_t K_h, int64_t V, int64_t n_occ, void* d_hidden, void* d_w,
                     int dw_fp32, int dtype, void* workspace, size_t workspace_bytes,
                     tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Per-occurrence clipped policy objective                                   */
/* ------------------------------------------------------------------------ */
/*
 * [TP] "The training-loop change is small": for PPO/GRPO every occurrence keeps its
 * own advantage, old log-probability, clipping rule, mask and weight (advantages
 * are not averaged before the clipped loss); [TT] §3.1 eq. 1 is the ratio-1 case
 * -A log p. With r_o = exp(logp_o - old_logp_o):
 *   loss[o]      = -w_o m_o min(r_o A_o, clip(r_o, 1 - eps_low, 1 + eps_high) A_o)
 *   grad_logp[o] = dL/dlogp_o = -w_o m_o A_o r_o where the unclipped term is the
 *                  minimum, 0 where the clipped one is (the input of tree_logprob_bwd)
 *   *loss_sum    = sum_o loss[o], summed in a fixed order (deterministic).
 * logp, old_logp, advantage: device fp32 [n_occ]; weight (fp32) and mask (uint8,
 * 0 = dropped) may be NULL (all ones). loss may be NULL unless loss_sum is wanted;
 * loss_sum: device fp32 scalar or NULL. 0 <= eps_low < 1, eps_high >= 0 finite.
 */
int tree_policy_loss(const float* logp, const float* old_logp, const float* advantage,
                     const float* weight, const uint8_t* mask, int64_t n_occ, float eps_low,
                     float eps_high, float* loss, float* grad_logp, float* loss_sum,
                     tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Partition-gateway attention                                               */
/* ------------------------------------------------------------------------ */
/*
 * [TT] §3.3 "Differentiable partition boundaries", Appendix B.2-B.5: a tree too
 * large for one pass is cut into partitions. A child partition C (T rows, its own
 * preorder subtree_end, local to C) attends to the keys/values its parent partition
 * accumulated up to the cut node -- the past, past_len rows -- under an additive
 * bias, 0 at the cut node's ancestors and -INFINITY elsewhere (eq. 15-16), and to
 * its own rows under the ordinary tree mask (eq. 14). Positions of C continue from
 * pos_offset (eq. 17): rotate q and the own rows of k with tree_rope beforehand.
 *
 * q, o, dout, dq: device [T, Hq, d]; k, v: device [past_len + T, Hkv, d], the past
 * rows first (the key/value cache a model holds); dk, dv: device [T, Hkv, d], the
 * gradients of C's own key/value rows (written). lse: device fp32 [Hq, T].
 * attn_bias: device fp32 [past_len], each 0 or -INFINITY (any other value sets the
 * device error word and is read as -INFINITY); may be NULL when past_len = 0.
 * dk_past, dv_past: device fp32 [past_len, Hkv, d]: the past rows' gradients are
 * ADDED to them in fp32 (B.5), so that the child partitions sharing one gateway sum
 * without bf16 rounding in between -- zero them before the first child.
 * Runs on the tensor-core kernels only: bf16, d = 128 (other
 * arguments: TREE_ERR_SHAPE / TREE_ERR_DTYPE). workspace: device, at least
 * tree_attn_gateway_workspace_size() bytes, 256-byte aligned. past_len = 0 is plain
 * tree attention (the same results as tree_attn_fwd / tree_attn_bwd).
 */
size_t tree_attn_gateway_workspace_size(int64_t past_len, int64_t T, int Hq, int Hkv, int d, int dtype);
int tree_attn_fwd_gateway(const void* q, const void* k, const void* v, void* o, float* lse,
                          const float* attn_bias, const int32_t* subtree_end, int64_t past_len,
                          int64_t T, int Hq, int Hkv, int d, int dtype, float softmax_scale,
                          void* workspace, size_t workspace_bytes, tree_stream_t stream);
int tree_attn_bwd_gateway(const void* q, const void* k, const void* v, const void* o,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          float* dk_past, float* dv_past, const float* attn_bias,
                          const int32_t* subtree_end, int64_t past_len, int64_t T, int Hq,
                          int Hkv, int d, int dtype, float softmax_scale, void* workspace,
                          size_t workspace_bytes, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Gated DeltaNet with tree state routing                                    */
/* ------------------------------------------------------------------------ */
/*
 * [TT] §3.2 "SSM Layers (GDN)", eq. 10, Appendix A.2: a GDN layer's recurrent state
 * is routed along the tree -- each node (chunk) starts from its parent node's end
 * state, a root node from zero -- so every row gets the state of an independent
 * per-branch pass. Per head, with state S [Dv, Dk]:
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
 * q, k: device [T, H, Dk]; v, o: device [T, H, Dv] (dtype); g (log decay), beta:
 * device fp32 [T, H]; q and k are used as given (normalising k or scaling q is the
 * caller's). node_start / node_end (inclusive) / node_parent: device int32
 * [n_nodes] from tree_pack_emit (nodes in preorder tiling [0, T), parents earlier; a
 * violation sets the device error word and leaves the outputs unwritten). Dk, Dv <=
 * 128, H <= 65535. fp32 arithmetic. workspace: device, >= tree_gdn_workspace_size()
 * bytes, 256-byte aligned (the sub-chunk table, the per-64-row-sub-chunk factors of
 * the chunked solution, and every sub-chunk's end state). Waits between the CTAs
 * that carry the state from a sub-chunk to the next are bounded (TREE_ERR_TIMEOUT in
 * the device error word; outputs then unspecified).
 */
size_t tree_gdn_workspace_size(int64_t T, int64_t n_nodes, int H, int Dk, int Dv);
int tree_gdn_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                 void* o, const int32_t* node_start, const int32_t* node_end,
                 const int32_t* node_parent, int64_t T, int64_t n_nodes, int H, int Dk, int Dv,
                 int dtype, void* workspace, size_t workspace_bytes, tree_stream_t stream);

/*
 * Backward of tree_gdn_fwd: the gradients of L = sum(dout * o) with respect to q, k,
 * v (dq, dk: device [T, H, Dk]; dv: device [T, H, Dv]; dtype, written) and to g and
 * beta (dg, dbeta: device fp32 [T, H], written). The state gradient flows back along
 * the same routing: a node's end-state gradient is the sum of the start-state
 * gradients of the nodes that continue from it (its next sub-chunk, or its children:
 * siblings share their parent's end state), summed in a fixed order, so the results
 * are reproducible run to run. dout: device [T, H, Dv] (dtype). The forward's states
 * are recomputed (the call needs only the forward's inputs). Other arguments as
 * tree_gdn_fwd; workspace: device, >= tree_gdn_bwd_workspace_size() bytes, 256-byte
 * aligned.
 */
size_t tree_gdn_bwd_workspace_size(int64_t T, int64_t n_nodes, int H, int Dk, int Dv);
int tree_gdn_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                 const void* dout, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                 const int32_t* node_start, const int32_t* node_end,
                 const int32_t* node_parent, int64_t T, int64_t n_nodes, int H, int Dk, int Dv,
                 int dtype, void* workspace, size_t workspace_bytes, tree_stream_t stream);

/*
 * tree_gdn_bwd without recomputing the forward: the sub-chunk factors, the delta-rule
 * corrections and the end states are taken from `workspace`, which must be the buffer
 * (>= tree_gdn_bwd_workspace_size() bytes) that the most recent tree_gdn_fwd on these
 * inputs ran with, on the same stream or synchronised since. Arguments and results as
 * tree_gdn_bwd, which it matches bit for bit. The forward marks the workspace with a
 * stamp of its shapes, dtype and input addresses; this call checks it on the device
 * and consumes it (a second call needs a new forward). On a mismatch -- another
 * workspace, other inputs or shapes, or no forward since the last use -- it schedules
 * nothing, sets TREE_ERR_DEVICE_CHECK in the device error word and leaves the outputs
 * unwritten. The stamp cannot see inputs changed in place between the two calls: they
 * must hold the forward's values.
 */
int tree_gdn_bwd_saved(const void* q, const void* k, const void* v, const float* g, const float* beta,
                       const void* dout, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                       const int32_t* node_start, const int32_t* node_end,
                       const int32_t* node_parent, int64_t T, int64_t n_nodes, int H, int Dk, int Dv,
                       int dtype, void* workspace, size_t workspace_bytes, tree_stream_t stream);

/* Test hook for the bounded waits of the GDN calls: the next tree_gdn_fwd or
 * tree_gdn_bwd call in this process withholds every publication of sub-chunk
 * `sub_chunk` (its index in preorder, -1 for none) and gives up any wait after
 * wait_seconds (0 < wait_seconds <= 2). Its successors' waits then run out: the call
 * ends with TREE_ERR_TIMEOUT in the device error word and unspecified outputs, and
 * the next call runs normally. TREE_ERR_INVALID_ARG for arguments out of range. */
int tree_gdn_test_withhold(int64_t sub_chunk, double wait_seconds);

/* ------------------------------------------------------------------------ */
/* Tree-correct causal depthwise conv1d (short convolution of SSM layers)    */
/* ------------------------------------------------------------------------ */
/*
 * [TT] §3.2 "(ii) Causal convolution", eq. 11 and Fig. 4: a causal conv of kernel
 * size K reads the K-1 tokens before each token; in the preorder serialisation
 * those rows may belong to a sibling branch, so the left context of a row is its
 * nearest ancestors (reaching past a short parent chunk into the grandparent),
 * zero above the root -- exactly what the row sees in a per-branch pass with zero
 * left padding. With a_0(i) = i and a_{m+1}(i) = parent_row[a_m(i)]:
 *   y[i, c] = bias[c] + sum_{m=0}^{K-1} w[c, K-1-m] * x[a_m(i), c]
 * (tap K-1 multiplies the row itself, tap 0 the farthest ancestor). No activation.
 *
 * x, y, dy, dx: device [T, C] in `dtype`, row-major, 16-byte aligned; w: device
 * [C, K] in `dtype`; bias: device [C] in `dtype` or NULL (no bias); C a multiple
 * of 8, 1 <= K <= 8. parent_row: device int32 [T] from tree_pack_emit (-1 for a
 * root, otherwise an earlier row). Arithmetic in fp32; y, dx rounded once.
 * A parent_row entry that is not an earlier row (or -1) sets the device error word
 * (TREE_ERR_DEVICE_CHECK) and is read as -1.
 */
int tree_conv1d_fwd(const void* x, const void* w, const void* bias, void* y,
                    const int32_t* parent_row, int64_t T, int C, int K, int dtype,
                    tree_stream_t stream);

/* Bytes of workspace tree_conv1d_bwd needs (per-tile partial sums of dw and
 * dbias, fp32); 0 for invalid sizes. */
size_t tree_conv1d_workspace_size(int64_t T, int C, int K);

/*
 * Gradients of L = sum(dy * y) for tree_conv1d_fwd: with D_m[j] the sum of dy over
 * the rows whose m-th ancestor is j (the descendants of j at depth m below it),
 *   dx[j, c]     = sum_m w[c, K-1-m] D_m[j, c]        (written in `dtype`)
 *   dw[c, K-1-m] = sum_j x[j, c] D_m[j, c]            (device fp32 [C, K], written)
 *   dbias[c]     = sum_i dy[i, c]                     (device fp32 [C], written)
 * dw and dbias may be NULL (not computed). The descendants are found from the
 * preorder intervals: subtree_end (device int32 [T]) and position_ids (device
 * int32 [T], depth of each row), both from tree_pack_emit. dw and dbias are summed
 * in a fixed order (deterministic). Entries inconsistent with a preorder forest
 * set the device error word. workspace: device, >= tree_conv1d_workspace_size(T,
 * C, K) bytes, 256-byte aligned. T = 0 writes zero dw and dbias.
 */
int tree_conv1d_bwd(const void* x, const void* w, const void* dy, void* dx, float* dw,
                    float* dbias, const int32_t* subtree_end, const int32_t* position_ids,
                    int64_t T, int C, int K, int dtype, void* workspace,
                    size_t workspace_bytes, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */
/* Synchronises `stream`, reads and clears the device error word of the current
 * device: TREE_OK, TREE_ERR_DEVICE_CHECK or TREE_ERR_TIMEOUT (a bounded
 * pipeline wait gave up; the kernel then returned early and its outputs are
 * unspecified), or TREE_ERR_CUDA if a CUDA error is pending. */
int tree_check_device_status(tree_stream_t stream);

/* Message of the last failure on this host thread ("" if none). Valid until the
 * next call into the library from the same thread. */
const char* tree_last_error(void);

/* Which kernel family a call with these arguments runs: 0 = CUDA-core fp32 kernels,
 * 1 = tcgen05 kind::f16 tensor-core kernels (bf16 operands), 2 = tcgen05 kind::tf32
 * tensor-core kernels with the two-term split. op: 0 attention forward, 1 attention
 * backward, 2 log-prob forward, 3 log-prob backward. */
int tree_kernel_path(int op, int dtype, int d);

/* Kernel launches this library has enqueued in this process (all devices, all
 * threads), for launch accounting by benchmarks. */
uint64_t tree_launch_count(void);

/* Kernel timing for benchmarks. With tree_kernel_timing(1), each attention call
 * brackets its main kernel with CUDA events on its stream (which = 0: the
 * forward's, 1: the backward's), and each conv1d call its kernels (2: forward,
 * 3: backward with its dw / dbias reduction); tree_kernel_last_ms(which) waits for the latest
 * bracket on the current device and returns its duration in ms, or -1 if there
 * is none. Off by default; leave it off while a stream is being captured. */
int tree_kernel_timing(int enable);
float tree_kernel_last_ms(int which);

/* Evaluates the FMA-pipe 2^x that the attention softmax uses for part of its
 * exponentials on x [n] (device fp32) into y [n] (device fp32), for tests against
 * the hardware exp2. Inputs below -125 give 2^-125. */
int tree_selftest_exp2(const float* x, float* y, int64_t n, tree_stream_t stream);

const char* tree_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TREE_ATTN_H_ */
