/*
 * gdnspec.h -- C ABI of the GB300 (sm_103a) library for speculative
 * verification and accepted-path commit of Gated DeltaNet (GDN) layers.
 *
 * Source of the method: "Pith review of SpecLA: Efficient Speculative
 * Decoding for Linear-Attention Models" (pith.science 7ERME3HB) -- "Core
 * claim" and "What carries the argument" (tree-masked factorized verifier,
 * factor buffering, the pending commit carried out by the next verification,
 * V-dimension tiling for chains) and the Referee Report's summary.  The
 * recurrence is the gated delta rule of "Gated Delta Networks: Improving
 * Mamba2 with Delta Rule", which that review cites:
 *
 *     S_t = alpha_t S_parent(t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t,
 *
 * applied along each draft node's own root-to-node path, starting from the
 * committed state S0.  S is d_v x d_k per (sequence, head), stored row-major
 * (row = value index).
 *
 * Conventions for every entry point
 *   - Every array argument is a DEVICE pointer owned by the caller, 16-byte
 *     aligned, densely packed in the layout stated.  The library never
 *     allocates device memory: factor buffers and workspaces are sized by
 *     gdn_factors_bytes / gdn_workspace_bytes and passed in.
 *   - Work is enqueued asynchronously on `stream` (0 = legacy default stream)
 *     of the current device, which must be an sm_103 GPU.
 *   - Shapes: 1 <= B, 1 <= H, 1 <= N <= 64 draft nodes per tree,
 *     d_k and d_v in {16, 32, ..., 256}.  B * H * N must fit in int32.
 *   - q/k/v element type: GDN_DTYPE_BF16 or GDN_DTYPE_F32.  alpha, beta, S,
 *     outputs and the buffered innovations are fp32.
 *   - Return value: GDN_OK, or a negative status for errors found on the host
 *     (bad shape, null or misaligned pointer, unsupported device, failed
 *     launch).  Errors found on the device (invalid parent_idx, invalid
 *     accepted path, a bounded wait that ran out) are recorded in a per-device
 *     error word and read back by gdn_last_error; kernels never trap.  After a
 *     device-side error the outputs of that call are unspecified.
 *   - Draft trees: parent_idx[b][t] is -1 (node hangs directly under the
 *     committed state) or an earlier node index (topological order).  Several
 *     -1 entries (a forest) are allowed; the arithmetic is the same.
 */
#ifndef GDNSPEC_H
#define GDNSPEC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define GDN_OK 0
#define GDN_ERR_ARG (-1)      /* bad shape, null or misaligned pointer, aliasing */
#define GDN_ERR_TREE (-2)     /* parent_idx[t] >= t or < -1 (device-detected) */
#define GDN_ERR_PATH (-3)     /* accepted path not root-first parent-chained (device-detected) */
#define GDN_ERR_TIMEOUT (-4)  /* a bounded device wait ran out (device-detected) */
#define GDN_ERR_CUDA (-5)     /* a CUDA runtime call or launch failed */
#define GDN_ERR_DEVICE (-6)   /* current device is not sm_103 */
#define GDN_ERR_CAPACITY (-7) /* request larger than a fixed on-device capacity (gdn_tree_verify_noalloc's
                                 scratch array) */

/* ---- q/k/v element types ------------------------------------------------ */
#define GDN_DTYPE_BF16 0
#define GDN_DTYPE_F32 1

/*
 * Factor buffer.  Verification writes, for every draft node, the compact
 * record the commit needs (review, "Core claim": the verifier keeps a small
 * record per draft token, and only the accepted tokens' records are applied):
 *
 *   delta  fp32  [B][H][N][d_v]   innovation delta_t = beta_t (v_t - alpha_t S_parent k_t)
 *   key    dtype [B][H][N][d_k]   k_t (same element type as the q/k/v inputs)
 *   g      fp32  [B][H][N]        cumulative log gate g_t = sum_{j on path(t)} log alpha_j
 *   parent int32 [B][N]           copy of parent_idx
 *
 * Sections are placed in this order, each starting on a 256-byte boundary.
 * With these, the state after accepting node a is
 *   S_a = e^{g_a} S0 + sum_{j on path(a)} e^{g_a - g_j} delta_j k_j^T.
 * gdn_factors_bytes writes the buffer size for a tree of N nodes.
 */
int gdn_factors_bytes(int B, int N, int H, int dk, int dv, int dtype, size_t* bytes);

/*
 * Workspace of the tree verifier: per-(sequence, head) coefficient tables of
 * the masked solve (review, "Core claim": A_tree = M_tree (.) (K_b K_a^T),
 * T_tree = solve_tril(I - A_tree)).  gdn_workspace_bytes writes its size;
 * contents are scratch, valid only during one call.
 */
int gdn_workspace_bytes(int B, int N, int H, int dk, int dv, size_t* bytes);

/*
 * Ancestor mask of each draft tree (review, "Core claim": the tree mask
 * M_tree that lets updates propagate only along ancestor paths).
 *   parent_idx int32 [B][N]
 *   mask       uint64 [B][N]: bit j of mask[b][t] set iff node j is a strict
 *              ancestor of node t (N <= 64)
 *   depth      int32 [B][N]: number of strict ancestors (roots have depth 0)
 * Invalid parent_idx -> GDN_ERR_TREE in the error word.
 */
int gdn_tree_mask(const int32_t* parent_idx, int B, int N, uint64_t* mask, int32_t* depth,
                  cudaStream_t stream);

/*
 * Tree-masked factorized verification (review, "Core claim" / "What carries
 * the argument": O = Qhat S0^T - Attn (W S0^T) + Attn U from the masked UT
 * solve).  One pass gives the output of every draft node, all computed from S0.
 *   q, k       dtype [B][N][H][d_k]
 *   v          dtype [B][N][H][d_v]
 *   alpha,beta fp32  [B][N][H]      gate in (0, 1], write strength
 *   parent_idx int32 [B][N]
 *   S0         fp32  [B][H][d_v][d_k]   committed state (read only)
 *   out        fp32  [B][N][H][d_v]     o_t for every node
 *   factors    gdn_factors_bytes(B,N,H,dk,dv,dtype) bytes, written
 *   workspace  gdn_workspace_bytes(B,N,H,dk,dv) bytes, scratch
 * out, factors and workspace must not overlap each other or the inputs.
 */
int gdn_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                    const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                    void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                    cudaStream_t stream);

/*
 * gdn_tree_verify without the workspace argument, for callers that cannot
 * allocate device memory: code running inside a host framework that owns all
 * device memory through its own pool and forbids raw cudaMalloc, and
 * latency-critical decode loops where an allocation and the device
 * synchronization it may imply are not acceptable.  (The paper has no
 * counterpart; this is a property of this library's interface.)
 *   Same arguments, layouts and results as gdn_tree_verify.  The workspace
 *   lives in a fixed 32 MiB scratch array inside the library, held by every
 *   GPU that loads the library until the process exits.  Shapes that run the
 *   single-kernel tensor-core verifier (bf16 q/k with d_k = d_v = 256) need
 *   no workspace and have no limit here.  For every other shape B * H *
 *   (workspace record of one (sequence, head)) must fit in the array -- at
 *   N = 64 that is up to 992 (sequence, head) pairs, e.g. B = 124 with H = 8;
 *   larger requests return GDN_ERR_CAPACITY without launching anything.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.  The call allocates nothing.
 *   All calls on a device share the array, which keeps the last call's
 *   contents (every entry is rewritten before it is read, so nothing needs
 *   clearing); calls whose kernels overlap on the GPU -- e.g. on two streams
 *   at once -- race on it.
 */
int gdn_tree_verify_noalloc(const void* q, const void* k, const void* v, int dtype,
                            const float* alpha, const float* beta, const int32_t* parent_idx,
                            const float* S0, float* out, void* factors, int B, int N, int H, int dk,
                            int dv, cudaStream_t stream);

/*
 * Chain verification with the state kept on chip and tiled along d_v
 * (review, "What carries the argument": a serial chain kernel with the
 * state cut into tiles along d_v).  The draft is a linear chain: node t hangs under t-1 and
 * node 0 under S0.  Same tensors and factor record as gdn_tree_verify
 * (the factor buffer's parent section receives -1, 0, 1, ..., N-2).
 */
int gdn_chain_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                     const float* beta, const float* S0, float* out, void* factors, int B, int N,
                     int H, int dk, int dv, cudaStream_t stream);

/*
 * Accepted-path commit from buffered factors, without snapshots or replay
 * (review, Referee Report summary: the state after the accepted tokens is
 * rebuilt from the per-token records, with no snapshot and no replay).
 *   S0            fp32 [B][H][d_v][d_k]   state the factors were verified from
 *   factors       written by a verify call with the same B, N, H, d_k, d_v, dtype
 *   accepted_path int32 [B][Lmax]: root-first accepted nodes, padded with -1;
 *                 path[b][0] must be a root, path[b][i] a child of path[b][i-1].
 *                 An all -1 row accepts nothing (S_new = S0, bit-identical).
 *   S_new         fp32 [B][H][d_v][d_k]; may equal S0 (in place)
 * 1 <= Lmax <= 64.  Invalid path -> GDN_ERR_PATH in the error word.
 */
int gdn_commit(const float* S0, const void* factors, const int32_t* accepted_path, int Lmax,
               float* S_new, int B, int N, int H, int dk, int dv, int dtype, cudaStream_t stream);

/*
 * Delayed state update carried out by the next verification (review, "Core
 * claim": the accepted path is applied to the state by the kernel that
 * verifies the following draft).  In one pass over the state tiles:
 *   S <- commit(S, prev_factors, prev_path)   (written back once, in place)
 *   then the new tree is verified from the committed S, as gdn_tree_verify.
 *   S            fp32 [B][H][d_v][d_k], in: state before the commit, out: committed
 *   prev_factors factor buffer of the previous verify (tree size N_prev)
 *   prev_path    int32 [B][Lmax] accepted path into the previous tree
 *   factors      factor buffer for the new tree (must not overlap prev_factors)
 * Other arguments as gdn_tree_verify.
 */
int gdn_commit_tree_verify(float* S, const void* prev_factors, int N_prev, const int32_t* prev_path,
                           int Lmax, const void* q, const void* k, const void* v, int dtype,
                           const float* alpha, const float* beta, const int32_t* parent_idx,
                           float* out, void* factors, void* workspace, int B, int N, int H,
                           int dk, int dv, cudaStream_t stream);

/* As gdn_commit_tree_verify, with the new draft a linear chain (gdn_chain_verify). */
int gdn_commit_chain_verify(float* S, const void* prev_factors, int N_prev,
                            const int32_t* prev_path, int Lmax, const void* q, const void* k,
                            const void* v, int dtype, const float* alpha, const float* beta,
                            float* out, void* factors, int B, int N, int H, int dk, int dv,
                            cudaStream_t stream);

/*
 * Full GDN layer decode step over B draft trees ("Pith review of SpecLA",
 * Referee Report, major comment 1: one GDN layer, h_v heads of d_k = d_v,
 * a four-tap causal depthwise conv, SiLU gate on the output; "Core
 * claim": every node sees the recurrence along its own root-to-node path).
 * For every node t of every tree, in one call on `stream`:
 *   Y_t   = W_in x_t = [q~ | k~ | v~ | z | a | b]_t            (bf16 GEMM, fp32)
 *   c_t   = sum_i conv_w[:, i] * u_i over the window u_0..u_3 = the pre-conv
 *           q~|k~|v~ rows of (great-grandparent, grandparent, parent, t); window
 *           positions above a root take the committed conv history (no bias,
 *           no activation)
 *   q_t, k_t = c_t's q and k parts L2-normalised per head; v_t = c_t's v part
 *   alpha_t = exp(-softplus(a_t)), beta_t = sigmoid(b_t)             (per head)
 *   o_t   = gated delta rule along path(t) from S (gdn_commit_tree_verify)
 *   out_t = W_o (o_t * SiLU(z_t))                      (bf16 GEMM, fp32 out)
 * The previous step's accepted path is committed first (delayed update): S
 * and the conv history move along prev_path using prev_record.
 *   X           bf16 [B][N][hidden]
 *   W_in        bf16 [2 H d_k + 2 H d_v + 2 H][hidden], row blocks q, k, v, z, a, b
 *   conv_w      fp32 [H (2 d_k + d_v)][4], tap 0 = oldest window position
 *   W_o         bf16 [hidden][H d_v]
 *   parent_idx  int32 [B][N], as gdn_tree_verify
 *   S           fp32 [B][H][d_v][d_k]; in: state before prev_path, out: committed
 *   conv_state  fp32 [B][3][H (2 d_k + d_v)], oldest row first; in/out like S
 *   prev_record the record written by the previous step (N_prev nodes per tree),
 *               with prev_path int32 [B][Lmax] (root first, -1 padded); both NULL
 *               when there is nothing to commit
 *   out         fp32 [B][N][hidden]
 *   record      gdn_layer_record_bytes bytes: this step's projections Y (fp32,
 *               row stride rounded up to 4 elements) and its factor record
 *               (fp32 keys); keep it until the next step's commit.  Must not
 *               overlap prev_record, workspace or out.
 *   workspace   gdn_layer_workspace_bytes bytes of intermediates (q, k, v,
 *               alpha, beta, o, the bf16 hi/lo terms of the gated output)
 * hidden a multiple of 64; H d_v a multiple of 64; d_k, d_v, N as gdn_tree_verify.
 * The caller owns every buffer; the call allocates nothing.  Errors: as
 * gdn_commit_tree_verify (GDN_ERR_TREE / GDN_ERR_PATH in the error word).
 */
int gdn_layer_record_bytes(int B, int N, int H, int hidden, int dk, int dv, size_t* bytes);
int gdn_layer_workspace_bytes(int B, int N, int H, int hidden, int dk, int dv, size_t* bytes);
int gdn_layer_tree_step(const void* X, const void* W_in, const float* conv_w, const void* W_o,
                        const int32_t* parent_idx, float* S, float* conv_state, const void* prev_record,
                        int N_prev, const int32_t* prev_path, int Lmax, float* out, void* record,
                        void* workspace, int B, int N, int H, int hidden, int dk, int dv,
                        cudaStream_t stream);

/*
 * Per-kernel timing of gdn_layer_tree_step (a measurement hook; the pages have
 * no counterpart).  events: host array of 6 cudaEvent_t handles created by the
 * caller (with timing enabled) on the device the layer runs on; n = 6 turns the
 * hook on, n = 0 (events ignored) turns it off.  While on, every
 * gdn_layer_tree_step call records, on its stream, events[i] just before its
 * kernel i (0 input GEMM, 1 conv, 2 tree verifier, 3 output gate, 4 output
 * GEMM) and events[5] after the last one, so cudaEventElapsedTime(events[i],
 * events[i + 1]) is kernel i's device time.  Process-wide; the caller keeps the
 * events alive while the hook is on and does not turn it on during stream
 * capture.  Other n, or a null handle, returns GDN_ERR_ARG.
 */
int gdn_layer_stage_events(void* const* events, int n);

/*
 * L GDN layers back to back over the same draft trees (layer-major
 * verification, "Pith review of SpecLA", "What carries the argument": the
 * layers are verified one after another, each streaming its own state).  Layer
 * l runs the layer step of gdn_layer_tree_step on input h_l with its own
 * weights, state, convolution history and records, on a residual stream:
 * h_0 = X, h_{l+1} = h_l + out_l in fp32 (entering each input projection as
 * two bf16 terms, hi + lo).  `out` (fp32 [B][N][hidden]) receives h_L.
 *   W_in, conv_w, W_o, S, conv_state, records, prev_records: host arrays of L
 *           device pointers, each as in gdn_layer_tree_step (prev_records and
 *           prev_path both NULL when there is nothing to commit)
 *   workspace  gdn_model_workspace_bytes bytes (one layer's workspace, the layer
 *           output and the residual stream in fp32 and as bf16 hi/lo terms)
 */
int gdn_model_workspace_bytes(int L, int B, int N, int H, int hidden, int dk, int dv, size_t* bytes);
int gdn_model_tree_step(int L, const void* X, const void* const* W_in, const float* const* conv_w,
                        const void* const* W_o, const int32_t* parent_idx, float* const* S, float* const* conv_state,
                        void* const* prev_records, int N_prev, const int32_t* prev_path, int Lmax, float* out,
                        void* const* records, void* workspace, int B, int N, int H, int hidden, int dk, int dv,
                        cudaStream_t stream);

/*
 * Per-token decoding of the same layer, for comparison with the tree step:
 * node t of every tree is decoded on its own (input projection at B rows,
 * its conv window, one delta-rule step from the parent's materialised state,
 * output gate, output projection), as a sequential decoder that keeps one
 * state per draft node would do ("Pith review of SpecLA", "Core claim": the
 * tree verifier replaces this node-by-node recurrence).  Calling it for
 * t = 0 .. N-1 in order yields the outputs of gdn_layer_tree_step.
 *   S0          fp32 [B][H][d_v][d_k] committed state (read only)
 *   conv_state  fp32 [B][3][H (2 d_k + d_v)] committed conv history (read only)
 *   S_nodes     fp32 [N][B][H][d_v][d_k]: the state after node t is written to
 *               S_nodes[t]; node t reads its parent's entry (S0 for a root)
 *   record, workspace: as gdn_layer_tree_step (only the projection rows and the
 *               intermediates are used); node t's projection row is written and its
 *               ancestors' rows, written by earlier calls, are read
 *   out         fp32 [B][N][hidden]: row t of every sequence is written
 * Other arguments as gdn_layer_tree_step.  0 <= t < N.
 */
int gdn_layer_token_step(const void* X, const void* W_in, const float* conv_w, const void* W_o,
                         const int32_t* parent_idx, const float* S0, const float* conv_state, float* S_nodes,
                         int t, float* out, void* record, void* workspace, int B, int N, int H, int hidden,
                         int dk, int dv, cudaStream_t stream);

/*
 * Chain-decomposed tree verification: serial within chains, parallel across
 * the chains that are ready ("Pith review of SpecLA", "What carries the
 * argument": a serial chain kernel with the state tiled along d_v, next to the
 * factorized tree form).  The tree is cut into chains (a chain starts at a
 * root or at a child of a node with two or more children and follows
 * only-children); chains whose parent chain is done run concurrently, each
 * token by token on state rows held in registers; a chain ending at a
 * branching node leaves its state rows in a slot for the chains below.  Same
 * tensors, outputs and factor record as gdn_tree_verify (so gdn_commit applies
 * to its factors).  Suited to deep, narrow trees.  Any valid tree runs: the
 * first 8 live branch states per tree are kept on chip, the rest spill to the
 * workspace.
 *   workspace  gdn_hybrid_workspace_bytes(B,N,H,dk,dv) bytes of device
 *              scratch, 16-byte aligned, not overlapping out or factors; may
 *              be NULL when that size is 0 (N <= 18).  Sized for the most
 *              branching nodes an N-node tree can have, (N - 1) / 2.
 * Returns GDN_ERR_ARG for bad shapes, pointers or overlaps (nothing launched);
 * an invalid parent_idx records GDN_ERR_TREE in the error word.
 */
int gdn_hybrid_workspace_bytes(int B, int N, int H, int dk, int dv, size_t* bytes);

int gdn_hybrid_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                           const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                           void* factors, void* workspace, int B, int N, int H, int dk, int dv, cudaStream_t stream);

/*
 * Confidence-guided pruning of B draft trees before verification ("Pith review
 * of SpecLA": confidence-guided tree pruning with a tree margin tau_tree and a
 * draft budget; the pages do not define them, the rule here is):
 *   score(t) = logp[t] + score(parent(t)), root first, fp32, where logp[t] is
 *              the drafter's log-probability of node t given its parent (<= 0)
 *   node t survives if score(t) >= max over its siblings (same parent, t
 *              included) of score minus tau, and its parent survives
 *   of the survivors the `budget` highest scores are kept (ties to the lower
 *              index), a set closed under ancestors; kept nodes keep their order
 *   parent_idx  int32 [B][N], topological (as gdn_tree_verify)
 *   logp        fp32 [B][N]
 *   new_index   int32 [B][N]: new number of each node, -1 if pruned
 *   new_parent  int32 [B][N]: parents of the kept nodes in their new numbering;
 *               entries from n_kept[b] on are -1
 *   n_kept      int32 [B]
 * tau >= 0 (may be +inf), budget >= 0.  Invalid parent_idx -> GDN_ERR_TREE in
 * the error word, outputs untouched.
 */
int gdn_prune_tree(const int32_t* parent_idx, const float* logp, float tau, int budget, int32_t* new_index,
                   int32_t* new_parent, int32_t* n_kept, int B, int N, cudaStream_t stream);

/*
 * Replay baselines: what tree verification and the factor-buffer commit
 * replace ("Pith review of SpecLA", "Core claim": tree verification against
 * replaying every root-to-leaf path; accepted-state recovery from buffered
 * factors against replaying the accepted tokens).  Same tensors and layouts
 * as gdn_tree_verify / gdn_commit; fp32 state throughout.
 *
 * gdn_replay_tree_verify: every leaf's root-to-leaf path is run token by token
 * from S0 and o_t is written for each node on it (a node shared by several
 * leaves is recomputed by each, with identical results).  No factor record.
 *
 * gdn_replay_commit: the accepted root-first path (int32 [B][Lmax], -1 padded,
 * validated against parent_idx) is run token by token from S0 and the final
 * state is written to S_new (which may equal S0).  Invalid path ->
 * GDN_ERR_PATH in the error word, S_new untouched.
 */
int gdn_replay_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                           const float* beta, const int32_t* parent_idx, const float* S0, float* out, int B,
                           int N, int H, int dk, int dv, cudaStream_t stream);
int gdn_replay_commit(const void* k, const void* v, int dtype, const float* alpha, const float* beta,
                      const int32_t* parent_idx, const float* S0, const int32_t* accepted_path, int Lmax,
                      float* S_new, int B, int N, int H, int dk, int dv, cudaStream_t stream);

/*
 * Snapshot baseline of state management ("Pith review of SpecLA", Figure 11:
 * the factor-buffer commit against keeping every draft node's state and
 * against replaying the accepted tokens).  Same tensors as gdn_tree_verify;
 * fp32 state throughout.
 *
 * gdn_snapshot_tree_verify: every node's state S_t = alpha_t S_p + delta_t k_t^T,
 * delta_t = beta_t (v_t - alpha_t S_p k_t), is built from its parent's stored state
 * (S0 above a root) and stored, node by node in index order; o_t = S_t q_t.
 *   S_nodes  fp32 [N][B][H][d_v][d_k], written (N times the state)
 * Invalid parent_idx -> GDN_ERR_TREE in the error word.
 *
 * gdn_snapshot_commit: S_new = S_nodes[a] for the last node a of the accepted
 * path (int32 [B][Lmax], root first, -1 padded, checked against parent_idx);
 * S_new = S0 for an empty path.  S_new may equal S0.  Invalid path ->
 * GDN_ERR_PATH in the error word, that sequence's S_new untouched.
 */
int gdn_snapshot_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                             const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                             float* S_nodes, int B, int N, int H, int dk, int dv, cudaStream_t stream);
int gdn_snapshot_commit(const float* S_nodes, const float* S0, const int32_t* parent_idx,
                        const int32_t* accepted_path, int Lmax, float* S_new, int B, int N, int H, int dk,
                        int dv, cudaStream_t stream);

/*
 * Tree verification of decay-gated linear attention (Mamba-2 / RetNet-style:
 * S_t = alpha_t S_parent(t) + beta_t v_t k_t^T, o_t = S_t q_t, no delta-rule
 * erasure) through the same kernels and factor record: the review of SpecLA
 * ("Axiom & Free-Parameter Ledger", editorial summary) names other
 * linear-attention families for the same verify/commit runtime.  Here A = 0,
 * T = I and the factor record holds delta_t = beta_t v_t with k_t, g_t and the
 * parents, so gdn_commit commits it unchanged.  Arguments as gdn_tree_verify.
 * (DeltaNet is gdn_tree_verify with alpha = 1.)
 */
int gdn_linear_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                           const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                           void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                           cudaStream_t stream);

/*
 * Gated linear attention (GLA: one gate per key channel, no delta-rule
 * erasure) over a draft tree, with its own factor record and commit (review of
 * SpecLA, editorial analysis: GLA is one of the recurrence families whose
 * per-token records the same verify / commit runtime carries).  Along each
 * node's root-to-node path from S0:
 *     S_t = S_parent(t) diag(alpha_t) + beta_t v_t k_t^T,    o_t = S_t q_t,
 * alpha_t in (0, 1]^{d_k}.  Tensors as gdn_tree_verify except
 *   alpha      fp32 [B][N][H][d_k]   per-channel gates
 * GLA factor record (gdn_gla_factors_bytes), sections 256-byte aligned:
 *   delta  fp32  [B][H][N][d_v]   beta_t v_t
 *   key    dtype [B][H][N][d_k]   k_t
 *   g      fp32  [B][H][N][d_k]   sum of log alpha_j over path(t), root first
 *   parent int32 [B][N]
 * so that the state after accepting node a is
 *   S_a = S0 diag(e^{g_a}) + sum_{j on path(a)} delta_j (k_j (.) e^{g_a - g_j})^T,
 * which gdn_gla_commit evaluates (arguments as gdn_commit; an all -1 path row
 * gives S_new = S0 bit-identical; an invalid path records GDN_ERR_PATH and
 * leaves that sequence's S_new untouched).  The verifier's workspace has its
 * own size, gdn_gla_workspace_bytes.  Invalid parent_idx -> GDN_ERR_TREE.
 */
int gdn_gla_factors_bytes(int B, int N, int H, int dk, int dv, int dtype, size_t* bytes);
int gdn_gla_workspace_bytes(int B, int N, int H, int dk, int dv, size_t* bytes);
int gdn_gla_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                        const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                        void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                        cudaStream_t stream);
int gdn_gla_commit(const float* S0, const void* factors, const int32_t* accepted_path, int Lmax,
                   float* S_new, int B, int N, int H, int dk, int dv, int dtype, cudaStream_t stream);

/*
 * Launch overlap between consecutive calls (process-wide switch, default off;
 * returns the previous setting).  When on, the first kernel of every call is
 * launched as a programmatic dependent of the kernel before it on the stream:
 * it starts streaming its state tiles and pending-commit factors (and may
 * write the committed state back) while that kernel finishes, and waits for it
 * before reading q/k/v/alpha/beta/parent_idx and before writing anything
 * else.  This hides launch and prologue latency in a
 * layer-major sweep ("Pith review of SpecLA", "What carries the argument":
 * layer-major verification keeps per-layer state streaming back to back).
 * Contract while on: the state S, S0, the accepted path and the factor
 * buffers of a call must not be read or written by the previous call on the
 * stream (whose kernels may still run) -- e.g. the calls of a sweep visit
 * different layers, each with its own state and factors, and the accepted
 * paths are written before the sweep starts.
 */
int gdn_set_launch_overlap(int enable);

/*
 * Waits for `stream`, returns the first device-side error recorded on the
 * current device since the last call (GDN_OK if none) and clears it.
 */
int gdn_last_error(cudaStream_t stream);

/* Static description of a status code. */
const char* gdn_strerror(int code);

/*
 * Limit of every bounded device wait, in nanoseconds, for the current device
 * (failure detection; the pages have no counterpart).  A kernel wait that has
 * not completed after this long records GDN_ERR_TIMEOUT in the error word and
 * the kernel winds down (its outstanding copies drained, tensor memory freed)
 * instead of hanging.  Default 1 s; 1e3 <= ns <= 6e10, else GDN_ERR_ARG.  The
 * value is written to device memory synchronously; set it between calls, not
 * while kernels that wait are running.
 */
int gdn_set_wait_limit_ns(unsigned long long ns);

/*
 * Self-test of that failure path: launches one thread that waits, through the
 * kernels' own bounded wait, on an mbarrier nothing arrives on, with no copy
 * or MMA outstanding.  After the wait limit it records GDN_ERR_TIMEOUT and
 * returns, so gdn_last_error(stream) then reports GDN_ERR_TIMEOUT and the
 * context remains usable.  Returns GDN_OK once launched.
 */
int gdn_selftest_stuck_wait(cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GDNSPEC_H */
