/*
 * spec_verify.h -- C ABI of the draft-tree verification step (tree attention, ratio-test
 * verification with residual resampling, KV compaction) for one GB300 (sm_103a) GPU.
 *
 * Sources (page title, section):
 *   [TREE]  "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码: flattened tree, the
 *           ancestor mask (a token sees itself and its ancestors), the forward call
 *           logits = llm.forward(draft_tree, tree_mask, position_ids, kvcache) and tree
 *           verification level by level.
 *   [RATIO] "推测解码 2026" (guijiagi.com), 数学基础：拒绝采样: accept with min(1, p/q), resample from
 *           relu(p - q) normalised, discard later candidates; 工程实践中的考量 / KV Cache管理:
 *           roll back the K/V of rejected candidates.
 *   [CSDN]  "【模型后训练与深度推理】9 推理加速：推测解码与级联推理", section 7.1 (alpha = min(1, p/q),
 *           residual norm(max(0, p - q)), output distributed as p), section 5 (interface: prompt,
 *           draft length, probability tensors, a boolean accept mask, accepted tokens).
 *   [SURV]  "万字综述 10+ 种 LLM 投机采样推理加速方案" (m.haoling.cc), 5.2 (tree-based parallel
 *           decoding through an attention mask), 4.3 (argmax sampling, temp = 0), 12.4.3
 *           (PagedAttention / FlashDecoding as the framework features to fit).
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the caller allocates
 *     and owns all buffers, including workspaces.  The library never allocates, frees or
 *     synchronises; each call enqueues kernels on `stream` and returns.
 *   - The return code covers argument validation and launch errors only.  Errors in DEVICE DATA
 *     (a bad parent index, a token id >= V, a block id out of range, ...) are OR-ed as SPEC_REQ_*
 *     bits into the caller's per-request int32 `req_status[B]`; such a request produces
 *     out_len = 0 / n_acc = -1 and is rolled back by spec_kv_compact.  No kernel traps.
 *   - Nodes of all requests are packed: request r owns global nodes
 *     node_offset[r] .. node_offset[r+1]-1 (CSR, node_offset has B+1 entries); node 0 of a request
 *     is its root (the last committed token, whose K/V is not cached yet); `parent` holds LOCAL
 *     indices with parent[root] = -1 and 0 <= parent[i] < i (BFS / topological order).
 *   - T_r = node_offset[r+1] - node_offset[r] includes the root; T_max (host) bounds every T_r and
 *     may not exceed SPEC_MAX_TREE (256).
 *   - Row-major buffers whose rows are read with 16-byte vector loads (logits, probabilities,
 *     Q, K/V, O) must start on 16-byte boundaries and have 16-byte-multiple row strides.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (pass 0 for the legacy default stream). */
typedef struct CUstream_st* spec_stream_t;

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, bad size or stride, tau < 0, ... */
  SPEC_ERR_UNSUPPORTED = 2,    /* a valid but unimplemented shape (e.g. bf16 head_dim != 128) */
  SPEC_ERR_CUDA = 3,           /* a CUDA launch / driver error (see spec_last_cuda_error) */
  SPEC_ERR_TIMEOUT = 4,        /* reserved for host-side waits; device waits report via bits */
  SPEC_ERR_BAD_INPUT_DATA = 5  /* reserved: data errors are reported per request, see below */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;
typedef enum { SPEC_DRAFT_LOGITS = 0, SPEC_DRAFT_PROBS = 1 } spec_draft_kind_t;
typedef enum {
  SPEC_SIBLING_RESIDUAL = 0,   /* default: child k is tested against the k-fold residual */
  SPEC_SIBLING_INDEPENDENT = 1, /* every sibling tested against p; resample from max(0, p - q) */
  SPEC_SIBLING_MULTI_DRAFT = 2  /* siblings from different draft models, each with its own q:
                                   draft_row[c] names the row CHILD c was drawn from */
} spec_sibling_rule_t;

/* Per-request data-error bits OR-ed into req_status[r]. */
#define SPEC_REQ_BAD_PARENT    1   /* parent[0] != -1 or parent[i] not in [0, i) */
#define SPEC_REQ_BAD_SIZE      2   /* T_r < 1, T_r > T_max, or node_offset not monotone / > N */
#define SPEC_REQ_BAD_TOKEN     4   /* a draft token id outside [0, V) */
#define SPEC_REQ_BAD_DRAFT_ROW 8   /* tau > 0 and a draft row read is outside [0, R): a node
                                      with children's, or under the multi-draft rule a drafted
                                      node's own */
#define SPEC_REQ_BAD_DEPTH     16  /* a root-to-node path longer than max_path */
#define SPEC_REQ_BAD_BLOCK     32  /* a needed block_table entry outside [0, num_blocks) */
#define SPEC_REQ_TIMEOUT       64  /* a bounded device-side wait gave up (the result is invalid) */

#define SPEC_MAX_TREE 256

/* ------------------------------------------------------------------------------------------
 * spec_tree_build  [TREE]
 * For each request: depth[i] = number of proper ancestors of node i (root 0);
 * pos_id[i] = prefix_len[r] + depth[i] (position ids adapted to the tree);
 * anc_mask row i (ceil(T_max/32) uint32 words, bit j of word j/32 = LOCAL node j) has bit j set
 * iff j == i or j is an ancestor of i -- one row of the page's mask table;
 * is_internal[i] = 1 iff node i has at least one child.
 *   parent [N] int32, node_offset [B+1] int32, prefix_len [B] int32: inputs (device).
 *   depth, pos_id [N] int32; anc_mask [N][ceil(T_max/32)] uint32; is_internal [N] uint8: outputs.
 *   req_status [B] int32: output; this call (re)initialises it (0 or a SPEC_REQ_* bit) and the
 *   later calls of the round OR their bits into it.
 * Requests with a data error get their outputs set to -1 / 0 and a SPEC_REQ_BAD_* bit.
 * Errors: SPEC_ERR_INVALID_ARG for null or inconsistent arguments (B < 1, N < 0, T_max outside
 * [1, 256]); SPEC_ERR_CUDA on a launch failure.
 * ------------------------------------------------------------------------------------------ */
spec_status_t spec_tree_build(const int32_t* parent, const int32_t* node_offset,
                              const int32_t* prefix_len, int32_t B, int32_t N, int32_t T_max,
                              int32_t* depth, int32_t* pos_id, uint32_t* anc_mask,
                              uint8_t* is_internal, int32_t* req_status, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_tree_rope_kv_write  [TREE]
 * The step before tree attention: rotary position embedding (RoFormer, Su et al. 2021, section
 * 3.2 -- the pages say only that position ids must follow the tree) of every tree node's q and
 * new k at its position id, and the node's K/V stored where spec_tree_attention reads it.
 * For node n = node_offset[r] + i at position m = pos_id[n] (prefix_len[r] + depth, from
 * spec_tree_build), pair j < rotary_dim/2 of each head row turns by m * base^(-2j/rotary_dim):
 *   (a, b) -> (a cos - b sin, a sin + b cos),
 * pair j being components (2j, 2j+1) when `interleaved` != 0 and (j, j + rotary_dim/2)
 * otherwise (the half-split layout of LLaMA-family checkpoints); components past rotary_dim are
 * copied unchanged.  Rotated q goes to q_out; rotated k and unchanged v go to logical slot
 * prefix_len[r] + i of the paged cache (row slot % block_size of block
 * block_table[r][slot / block_size]).  Arithmetic: angle formed and reduced modulo 2 pi in fp64,
 * rotation in fp32, one rounding to `dtype`.
 * Layouts (element type `dtype`, contiguous, 16-byte aligned): q_in, q_out [N][H_q][head_dim]
 * (q_out == q_in rotates in place; partial overlap is not allowed); k_new, v_new
 * [N][H_kv][head_dim]; k_cache, v_cache [num_blocks][H_kv][block_size][head_dim] (one layer);
 * block_table [B][max_blocks_per_req], prefix_len [B], node_offset [B+1], pos_id [N] int32.
 * Data errors: nodes of a request with req_status[r] != 0 (e.g. from spec_tree_build) are not
 * touched; a request any of whose tree slots maps outside [0, num_blocks) gets
 * SPEC_REQ_BAD_BLOCK and none of its nodes is written.
 * Errors: SPEC_ERR_INVALID_ARG (null / misaligned pointers, bad sizes, rotary_dim odd or outside
 * [2, head_dim], base not positive and finite); SPEC_ERR_UNSUPPORTED when a rotated pair would
 * straddle 16-byte vectors (half-split: rotary_dim/2 must be a multiple of 8 bf16 / 4 fp32
 * elements; interleaved: rotary_dim a multiple of 8 / 4) or rotary_dim > 256; SPEC_ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  spec_dtype_t dtype;
  int32_t B, N, H_q, H_kv, head_dim, rotary_dim;
  int32_t interleaved;         /* 0: pairs (j, j + rotary_dim/2); 1: pairs (2j, 2j+1) */
  int32_t block_size, num_blocks, max_blocks_per_req;
  double base;                 /* e.g. 10000 (LLaMA-2), 500000 (LLaMA-3), 1e6 (Qwen2) */
  const void* q_in;
  void* q_out;
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* node_offset;
  const int32_t* pos_id;
  int32_t* req_status;
} spec_rope_params;

spec_status_t spec_tree_rope_kv_write(const spec_rope_params* p, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_tree_build_rope_kv_write  [TREE]
 * spec_tree_build and spec_tree_rope_kv_write in one launch: the tree outputs of
 * spec_tree_build (same arguments, same results), then -- for every request the tree build
 * accepts -- the rotary embedding and K/V slot write of spec_tree_rope_kv_write at
 * pos = prefix_len + depth, described by `rope` (host pointer; its B and N must equal this
 * call's, and its node_offset, prefix_len, pos_id and req_status must be NULL or this call's
 * buffers).  req_status[r] ends as spec_tree_build's bits, or SPEC_REQ_BAD_BLOCK for a valid
 * tree with a slot outside the pool (nothing of that request is then written to q_out or the
 * cache); the results equal the two calls made in sequence.
 * Errors: those of the two calls.
 * ------------------------------------------------------------------------------------------ */
spec_status_t spec_tree_build_rope_kv_write(const int32_t* parent, const int32_t* node_offset,
                                            const int32_t* prefix_len, int32_t B, int32_t N,
                                            int32_t T_max, int32_t* depth, int32_t* pos_id,
                                            uint32_t* anc_mask, uint8_t* is_internal,
                                            int32_t* req_status, const spec_rope_params* rope,
                                            spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_tree_attention  [TREE], [SURV 5.2, 12.4.3]
 * O[n][h] = sum_j softmax_j(scale * q[n][h] . k_j) v_j over the logical KV slots
 *   j in {0 .. P_r-1} U {P_r + a : a == i or a is an ancestor of i}
 * for node n = node_offset[r] + i.  The caller has written node a's K/V into logical slot
 * P_r + a before the call.  Logical slot s of request r is row s % block_size of physical block
 * block_table[r][s / block_size].  Query head h reads KV head h / (H_q / H_kv).
 * Layouts (element type `dtype`, contiguous, 16-byte aligned):
 *   q [N][H_q][head_dim]; k_cache, v_cache [num_blocks][H_kv][block_size][head_dim] (one layer);
 *   o [N][H_q][head_dim]; lse [N][H_q] fp32 (natural log of the softmax denominator of the
 *   scaled scores) or NULL; block_table [B][max_blocks_per_req] int32; prefix_len [B];
 *   node_offset [B+1]; anc_mask from spec_tree_build; req_status [B] in/out.
 * Paths: dtype BF16 runs on the tcgen05 tensor cores (TMA-staged paged tiles, scores and output
 * accumulated in TMEM) and requires head_dim == 128, block_size == 16 and
 * H_q / H_kv in {1, 2, 4, 8, 16}; dtype F32 runs a CUDA-core kernel (head_dim <= 128,
 * multiple of 4).  Long KV ranges are split across CTAs and merged by log-sum-exp in
 * `workspace` (spec_attention_workspace_size bytes, 256-byte aligned, caller-owned, contents
 * need not be initialised).  scale <= 0 selects 1/sqrt(head_dim).
 * Errors: SPEC_ERR_INVALID_ARG (null / misaligned pointers, inconsistent sizes, too-small
 * workspace), SPEC_ERR_UNSUPPORTED (a shape outside the paths above), SPEC_ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  spec_dtype_t dtype;
  int32_t B, N, T_max;
  int32_t H_q, H_kv, head_dim;
  int32_t block_size;          /* tokens per KV block */
  int32_t num_blocks;          /* physical blocks in the pool (bounds check) */
  int32_t max_blocks_per_req;  /* row stride of block_table */
  float scale;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* node_offset;
  const uint32_t* anc_mask;
  void* o;
  float* lse;
  int32_t* req_status;
} spec_attn_params;

size_t spec_attention_workspace_size(const spec_attn_params* p);
spec_status_t spec_tree_attention(const spec_attn_params* p, void* workspace, size_t ws_bytes,
                                  spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_verify  [RATIO], [CSDN 7.1, 7.2, 5], [TREE], [SURV 4.3]
 * p_i = softmax(target[i] / tau), q_i = softmax(draft[draft_row[i]] / tau) (draft logits) or the
 * given row (draft probabilities).  Walk from the root; at node i test its children c in
 * increasing index with u_acc = uniforms[c][0]:
 *   SIBLING_RESIDUAL: after k rejected siblings the target is R_k = max(0, p_i - C_k q_i),
 *     C_0 = 0, N_k = sum R_k, C_{k+1} = C_k + N_k; accept iff u_acc < R_k(tok)/(N_k q_i(tok))
 *     (k = 0: p/q, the pages' rule);
 *   SIBLING_INDEPENDENT: accept iff u_acc < p_i(tok)/q_i(tok) for every sibling;
 *   SIBLING_MULTI_DRAFT ([SURV 5.1] a group of small models predicting together; [TREE]
 *     merge-based trees from k small models): child c carries its own q_c = softmax(
 *     draft[draft_row[c]] / tau) -- draft_row is indexed by the CHILD, and every non-root node
 *     needs one (tau > 0).  The running target starts as R_0 = p_i, N_0 = 1; child j is
 *     accepted iff u_acc < R_{j-1}(tok)/(N_{j-1} q_c(tok)), and a rejection gives
 *     R_j = max(0, R_{j-1} - N_{j-1} q_c), N_j = sum R_j (the pages' norm(max(0, r - q))
 *     applied sibling after sibling); all rejected: the final token is drawn from R_k.  Needs
 *     two fp32 rows of ceil(V/64)*64 floats per request in the workspace (included in
 *     spec_verify_workspace_size); spec_verify_noalloc refuses it (SPEC_ERR_UNSUPPORTED);
 *   tau == 0: accept iff tok == argmax p_i (lowest id on ties).
 * On acceptance descend to c.  The walk stops at a leaf (the final token is a bonus draw from
 * p_leaf with u_samp = uniforms[leaf][1]) or when every child is rejected (the final token is
 * drawn from the normalised residual with u_samp of that node; from p if the residual mass is
 * 0); tau == 0 takes argmax p instead.  Draws use the inverse CDF over ascending token id: the
 * smallest x with sum_{y<=x} w(y) > u * sum_y w(y).  Randomness is never generated inside.
 * Outputs per request r (row stride max_path): path[r][0..n_acc] = accepted local node ids
 * (root first), out_tokens[r][0..n_acc] = accepted draft tokens then the final token,
 * out_len[r] = n_acc + 1, rejections[r] = rejected children on the walk; unused entries -1.
 * Layouts: target [N][target_ld] (logits_dtype), draft [R][draft_ld] (logits_dtype for
 * logits, fp32 for probabilities), rows 16-byte aligned; draft_row, tokens, parent, depth [N]
 * int32 (depth from spec_tree_build); is_internal [N] uint8; uniforms [N][2] fp32.
 * workspace: spec_verify_workspace_size bytes (256-byte aligned, caller-owned).
 * Errors: SPEC_ERR_INVALID_ARG (null / misaligned pointers, V < 1, ld < V, tau < 0 or not
 * finite, max_path < 1, small workspace), SPEC_ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  spec_dtype_t logits_dtype;
  spec_draft_kind_t draft_kind;
  spec_sibling_rule_t sibling_rule;
  int32_t B, N, R, V;
  int64_t target_ld, draft_ld;   /* row strides in elements */
  int32_t T_max, max_path;
  float tau;
  const void* target;
  const void* draft;
  const int32_t* draft_row;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* node_offset;
  const int32_t* depth;
  const uint8_t* is_internal;
  const float* uniforms;
  int32_t* req_status;
  int32_t* out_tokens;
  int32_t* out_len;
  int32_t* path;
  int32_t* n_acc;
  int32_t* rejections;           /* may be NULL */
  int32_t verify_path;           /* SPEC_VERIFY_PATH_AUTO (0, the default), _SPLIT or _WALK */
} spec_verify_params;

/* verify_path -- no counterpart on the pages: which of the library's forms of the same
 * computation this call launches.
 *   SPEC_VERIFY_PATH_AUTO (0, what a zero-initialised struct asks for): calls with the residual
 *     or independent sibling rule (or tau == 0), T_max <= 32 and
 *     T_max * S_t + (T_max - 1) * S_d <= 200 KiB run as one cluster launch (up to 8 CTAs per
 *     request, each holding its share of the request's rows in shared memory), with
 *     S_t / S_d = ceil(ceil(V / 8) / 8) * 8 * the target / draft element size (S_d = 0 at
 *     tau == 0); the others with those rules and V >= 65536 run the walk form, every other call
 *     the two-launch form;
 *   SPEC_VERIFY_PATH_SPLIT: always the two-launch form (a row statistics kernel for every
 *     internal node's rows, then a walk kernel with a cluster of CTAs per request);
 *   SPEC_VERIFY_PATH_WALK: the walk kernel alone, which forms the statistics (max and sum, or
 *     argmax at tau == 0) of the nodes it visits, one pass over their two rows each, instead of
 *     reading every internal node's rows first (the multi-draft rule always runs the two-launch
 *     form).
 * All forms give the same outputs except where fp32 rounding of the vocabulary sums decides:
 * a ratio test or a draw whose uniform lies within about 1e-6 of its boundary.  The choice is
 * per call: the library keeps no process-wide setting.  Any other value: SPEC_ERR_INVALID_ARG. */
#define SPEC_VERIFY_PATH_AUTO  0
#define SPEC_VERIFY_PATH_SPLIT 1
#define SPEC_VERIFY_PATH_WALK  2

size_t spec_verify_workspace_size(const spec_verify_params* p);
spec_status_t spec_verify(const spec_verify_params* p, void* workspace, size_t ws_bytes,
                          spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_verify_noalloc -- no counterpart on the pages; an addition for callers that may not
 * allocate device memory (an engine that reserves its whole memory budget up front and forbids
 * allocation while serving, or a plugin that is handed only tensors and a stream).
 * Same inputs, outputs and results as spec_verify, but the workspace is a fixed array in device
 * memory that belongs to this library (every GPU that loads the library keeps it until the
 * process exits), so the caller passes none and nothing is allocated.
 * Limits: N <= 32768 tree nodes and R <= 32768 draft rows per call; larger batches return
 * SPEC_ERR_UNSUPPORTED (use spec_verify with a caller-owned workspace instead).
 * The first call on each device looks up the array's device address with that device current;
 * make that first call before any stream capture.  Later calls look it up again unless their
 * stream is being captured, so a device reset between calls is safe.  All calls share the one
 * array: calls whose kernels overlap on the GPU (other streams, other host threads on the same
 * device) race.  The multi-draft sibling rule with tau > 0 is refused (SPEC_ERR_UNSUPPORTED).
 * Errors: as spec_verify, plus SPEC_ERR_UNSUPPORTED for sizes beyond the limits above and
 * SPEC_ERR_CUDA if the address lookup fails.
 * ------------------------------------------------------------------------------------------ */
spec_status_t spec_verify_noalloc(const spec_verify_params* p, spec_stream_t stream);


/* ------------------------------------------------------------------------------------------
 * spec_kv_compact  [RATIO: KV Cache管理], [CSDN 4]
 * Commits the accepted path and rolls back the rest, in place, for every layer and KV head,
 * K and V: new[P_r + d] = old[P_r + path[r][d]] for d = 0 .. n_acc[r] (gather semantics: every
 * source is read as it was before the call), i.e. the cache sequential decoding of the accepted
 * path would hold.  new_kv_len[r] = P_r + n_acc[r] + 1 (the final token has no K/V yet);
 * blocks_in_use[r] = ceil(new_kv_len / block_size); slot_map[r][d] = (src, dst) logical slots,
 * (-1, -1) past n_acc.  A request with req_status != 0 or n_acc < 0 is rolled back entirely
 * (new_kv_len = P_r, nothing copied).  Slots past new_kv_len are released, not cleared.
 * Layouts: k_cache, v_cache point at layer 0 of [num_layers] x [num_blocks][H_kv][block_size]
 * [head_dim] with `layer_stride` elements between layers; head_dim * element size must be a
 * multiple of 16 bytes.  path [B][max_path], n_acc [B] as written by spec_verify;
 * slot_map [B][max_path][2], new_kv_len [B], blocks_in_use [B] int32 outputs.
 * Errors: SPEC_ERR_INVALID_ARG, SPEC_ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  spec_dtype_t dtype;
  int32_t B, H_kv, head_dim, block_size, num_blocks, max_blocks_per_req, num_layers, max_path;
  int64_t layer_stride;
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* path;
  const int32_t* n_acc;
  int32_t* req_status;
  int32_t* new_kv_len;
  int32_t* slot_map;
  int32_t* blocks_in_use;
} spec_compact_params;

spec_status_t spec_kv_compact(const spec_compact_params* p, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_verify_compact -- spec_verify followed by spec_kv_compact, in one call: same inputs,
 * outputs and results as the two calls in that order.  When the verification takes its
 * one-launch form (see verify_path above) the compaction runs inside that launch (one
 * kernel for both); otherwise spec_kv_compact is launched after it.  The compaction reads the
 * verification's own results, so c->path, c->n_acc, c->req_status must be v->path, v->n_acc,
 * v->req_status, with c->B == v->B and c->max_path == v->max_path.
 * Errors: as spec_verify and spec_kv_compact, plus SPEC_ERR_INVALID_ARG when c is NULL or does
 * not match v as above.
 * ------------------------------------------------------------------------------------------ */
spec_status_t spec_verify_compact(const spec_verify_params* v, const spec_compact_params* c,
                                  void* workspace, size_t ws_bytes, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Building the draft tree on the device  [TREE 草稿树的生成, 动态草稿长度]
 * EAGLE-2 expands, level by level, only the K most probable leaves of the newest level (a
 * leaf's score is the sum of the draft log-probabilities along its path, log q =
 * log_softmax(draft_row / tau)[token]); each expansion adds the K most probable tokens of the
 * expanded node's draft row.  ECHO then keeps a batch-wide budget of K_max tokens: every root
 * and the K_max - B best non-root candidates of the batch.  The draft model's forward, which
 * turns the chosen candidates into draft rows, is the caller's.
 * Candidate pool (caller-owned device arrays, request r's candidates at [r * cap, r * cap +
 * count[r])): parent (candidate index, -1 for the root), token, depth, score (fp32), row (the
 * draft row its expansion produced, -1 if never), count.  cap <= 256.
 * Ordering everywhere: by score (or log-probability) descending, ties to the lower candidate
 * index / token id, then (ECHO) the lower request.  Selections compare the fp32 scores exactly.
 * A drafting round: spec_draft_init; for level = 1 .. depth: spec_draft_expand_select, the
 * caller's draft forward for the listed candidates, spec_draft_topk_append; then
 * spec_echo_select_pack, whose outputs feed spec_tree_build / spec_verify (draft_row indexes
 * the rows the caller produced, numbered row_base + r * K + j by the append calls).
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  int32_t B, cap;
  int32_t* parent;   /* [B][cap] */
  int32_t* token;    /* [B][cap] */
  int32_t* depth;    /* [B][cap] */
  float* score;      /* [B][cap] */
  int32_t* row;      /* [B][cap] */
  int32_t* count;    /* [B] */
} spec_draft_pool;

/* Pool entry 0 of request r = the root (root_tokens[r]), count = 1. */
spec_status_t spec_draft_init(const spec_draft_pool* pool, const int32_t* root_tokens,
                              spec_stream_t stream);

/* The candidates to expand at `level` (1: the root; else the K best of depth level - 1), in
 * increasing candidate index: expand[r][j], j < K, -1 past the chosen ones.  Grows count[r] by
 * K per chosen candidate; if the pool cannot hold that many, fewer are chosen and req_status[r]
 * (may be NULL) gets SPEC_REQ_BAD_SIZE.  1 <= K <= 16. */
spec_status_t spec_draft_expand_select(const spec_draft_pool* pool, int32_t level, int32_t K,
                                       int32_t* expand, int32_t* req_status,
                                       spec_stream_t stream);

/* For every expand[r][j] >= 0: the K most probable tokens of draft row r * K + j of `rows`
 * ([B * K][ld], dtype F32 / BF16 logits, 16-byte aligned rows, V <= ld), log q =
 * x / tau - logsumexp(row / tau) (one streaming read of the row), appended as the candidate's
 * children in that order with score = its score + log q, depth = level; the candidate's row
 * becomes row_base + r * K + j.  Call after spec_draft_expand_select of the same level.
 * req_status (may be NULL) gets SPEC_REQ_TIMEOUT if the launch's bounded wait ran out (only
 * under the testing hook below); that expansion's children then carry token -1 and score -inf. */
spec_status_t spec_draft_topk_append(const spec_draft_pool* pool, int32_t level, int32_t K,
                                     const int32_t* expand, spec_dtype_t dtype, const void* rows,
                                     int64_t ld, int32_t V, float tau, int32_t row_base,
                                     int32_t* req_status, spec_stream_t stream);

/* Testing only: with chunk >= 0, the following spec_draft_topk_append launches on the current
 * device wait (bounded, about a second) for a device flag that nothing sets, so they run out
 * their wait and report SPEC_REQ_TIMEOUT for those requests, as a lost read would, with
 * children of token -1 and score -inf; -1 restores normal operation.  Synchronous (a
 * host-to-device symbol copy). */
spec_status_t spec_debug_draft_copy_stall(int32_t chunk);

/* ECHO selection and packing: node_offset [B+1]; parent (local, -1 for roots), tokens, depth,
 * draft_row (the node's row if one of its children was kept, else -1) and source (candidate
 * index, may be NULL), each with room for min(K_max, B * cap) entries; N = node_offset[B].
 * Kept candidates stay in candidate order (parents first), so the output is a valid tree in
 * the layout spec_tree_build reads.  workspace: spec_echo_workspace_size(B, cap) bytes,
 * 256-byte aligned. */
size_t spec_echo_workspace_size(int32_t B, int32_t cap);
spec_status_t spec_echo_select_pack(const spec_draft_pool* pool, int32_t K_max,
                                    int32_t* node_offset, int32_t* parent, int32_t* tokens,
                                    int32_t* depth, int32_t* draft_row, int32_t* source,
                                    void* workspace, size_t ws_bytes, spec_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* spec_status_string(spec_status_t status);

/* The cudaError_t (as int) behind the most recent SPEC_ERR_CUDA on this thread, 0 if none. */
int spec_last_cuda_error(void);

/* No counterpart on the pages: how many kernels this library has enqueued in this process, all
 * threads and devices together (a launch made while a stream is captured counts once, when it
 * is captured; replays of the graph are not launches of the library).  Diagnostics only. */
uint64_t spec_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
