/*
 * jf.h -- C ABI of the GB300 (sm_103a) tree-speculative-decoding hot path:
 *   tree-causal attention mask  ->  tree-causal paged attention  ->  greedy tree verify.
 *
 * Source of the operations: "JetFlow: Breaking the Scaling Ceiling of Speculative
 * Decoding with Parallel Tree Drafting" (gist.science explainer, technical summary §2
 * "Method" -- tree-causal attention mask, branch factorisation, best-first tree
 * construction; §3 -- paged attention kernel with tree-mask staging used for tree
 * verification; §4 -- accepted tokens tau), and the qxai.app commentary on the same
 * paper (section "まず、何が問題なのか": the large model checks the drafted candidates
 * together and keeps the part it agrees with).
 *
 * Conventions shared by every call:
 *  - Every pointer argument except `stream` is a DEVICE pointer owned by the caller;
 *    the library never frees, keeps or allocates caller memory.  Scalars are host values.
 *  - Calls only enqueue kernels on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and return; they never synchronise.  Several calls may be captured in a
 *    CUDA graph.
 *  - Host-visible problems (null pointer, unsupported size, misalignment, small
 *    workspace) are returned synchronously and nothing is launched.
 *  - Data-dependent problems (a malformed tree, a page id outside the pool, a token
 *    outside the vocabulary, a prefix longer than the block table allows) are OR-ed as
 *    JF_DEVERR_* bits into *dev_err (a device int32 the caller zeroes and reads after
 *    its next synchronisation; may be NULL to skip reporting).  The affected outputs are
 *    then unspecified, but every access stays in bounds.  No kernel traps or asserts.
 *  - A kernel wait that exceeds its time limit (about one second) sets
 *    JF_DEVERR_TIMEOUT and the kernel returns instead of hanging.
 *  - Node numbering: parent[b][0] == -1 (the root) and 0 <= parent[b][i] < i.
 */
#ifndef JF_H_
#define JF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* jf_stream_t; /* identical to cudaStream_t */

typedef enum {
  JF_OK = 0,
  JF_ERR_INVALID_ARGUMENT = 1,    /* null pointer, non-positive size, bad dtype      */
  JF_ERR_INVALID_TREE = 2,        /* reserved: tree errors are reported on device      */
  JF_ERR_UNSUPPORTED = 3,         /* valid but unsupported shape (see each call)       */
  JF_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes below the *_workspace_size value  */
  JF_ERR_CUDA = 5,                /* a CUDA runtime call or kernel launch failed       */
  JF_ERR_TIMEOUT = 6,             /* reserved: timeouts are reported on device         */
  JF_ERR_MISALIGNED = 7,          /* a pointer is not 16-byte aligned where required   */
  JF_ERR_SCRATCH_CAPACITY = 8     /* sizes exceed the static scratch of a *_static call */
} jf_status;

typedef enum { JF_DTYPE_BF16 = 0, JF_DTYPE_F32 = 1 } jf_dtype;

/* Bits OR-ed into *dev_err. */
#define JF_DEVERR_BAD_PARENT 0x1 /* parent[0] != -1 or parent[i] outside [0, i)         */
#define JF_DEVERR_BAD_PAGE 0x2   /* block_table entry outside [0, num_pages)            */
#define JF_DEVERR_BAD_PREFIX 0x4 /* prefix_len < 0 or prefix_len + N > max_pages * page */
#define JF_DEVERR_BAD_TOKEN 0x8  /* draft token (non-root node) outside [0, V)          */
#define JF_DEVERR_TIMEOUT 0x10   /* an in-kernel wait gave up after its time limit      */
#define JF_DEVERR_BAD_PATH 0x20  /* accepted path / length malformed (KV compaction)     */
#define JF_DEVERR_BAD_TREE_LEN 0x40 /* tree_len[b] outside [1, N], or a bad packed span   */

/* Largest tree (nodes per sequence) any call accepts. */
#define JF_MAX_NODES 4096

/* Human-readable name of a jf_status value (static storage, never NULL). */
const char* jf_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int jf_version(void);

/*
 * jf_build_tree_mask -- tree-causal attention mask (explainer §2, "Tree-Causal Attention
 * Mask": a draft node attends to the prefix and to its own ancestors, never to its
 * descendants or to unrelated sibling branches).
 *
 *   parent     int32 [B][N]   parent[b][0] = -1, 0 <= parent[b][i] < i.
 *   prefix_len int32 [B]      P_b, number of prefix tokens before the tree.
 *   mask       uint64 [B][N][W], W = ceil(N / 64): bit (j & 63) of word (j >> 6) of row
 *                             (b, i) is 1 iff node j is node i or an ancestor of i.
 *                             Bits at j >= N are 0.
 *   depth      int32 [B][N]   number of ancestors of i (root: 0).  May be NULL.
 *   pos        int32 [B][N]   position id P_b + depth[b][i].          May be NULL.
 *   dev_err    int32 [1]      JF_DEVERR_BAD_PARENT on a malformed tree. May be NULL.
 * Limits: 1 <= N <= JF_MAX_NODES, B >= 1.  mask must be 8-byte aligned.
 */
jf_status jf_build_tree_mask(const int32_t* parent, const int32_t* prefix_len, int32_t B,
                             int32_t N, uint64_t* mask, int32_t* depth, int32_t* pos,
                             int32_t* dev_err, jf_stream_t stream);

/*
 * Bytes of device workspace jf_tree_attention and jf_tree_attention_ragged need for these
 * sizes on the CURRENT device (split-KV partial results).  0 means no workspace is needed.
 * Returns (size_t)-1 if the sizes are unsupported or the device cannot be queried.
 */
size_t jf_tree_attention_workspace_size(int32_t B, int32_t N, int32_t Hq, int32_t Hkv,
                                        int32_t D, int32_t max_pages, int32_t page_size);

/*
 * jf_tree_attention -- tree-causal paged attention (explainer §2 mask and branch
 * factorisation q(pi(v)|x) = prod_{u in pi(v)} q(y_u | x, h_x, pi_{<u}); §3 paged
 * attention kernel for tree verification).  For every sequence b, query head h and
 * node i, with kv-head g = h / (Hq / Hkv):
 *     visible keys S = {0 .. P_b-1} u {P_b + j : bit j of mask[b][i] is set}
 *     out[b][i][h] = sum_{t in S} softmax_t(scale * q . k_t) v_t
 *     lse[b][h][i] = log sum_{t in S} exp(scale * q . k_t)      (natural log)
 * Key/value t of sequence b is row (page = block_table[b][t / page_size],
 * slot = t % page_size, head g) of the paged pool; the N tree nodes' keys/values sit at
 * logical positions P_b .. P_b + N - 1, right after the prefix.
 *
 *   q            bf16 [B][N][Hq][D]                    (RoPE already applied)
 *   k_cache      bf16 [num_pages][page_size][Hkv][D]
 *   v_cache      bf16 [num_pages][page_size][Hkv][D]
 *   block_table  int32 [B][max_pages]; entries past ceil((P_b + N) / page_size) are
 *                never read.
 *   prefix_len   int32 [B]
 *   mask         uint64 [B][N][W] as written by jf_build_tree_mask.
 *   scale        softmax scale (usually 1 / sqrt(D)).
 *   out          bf16 [B][N][Hq][D] (written, round-to-nearest-even).
 *   lse          float [B][Hq][N] or NULL.
 *   workspace    device buffer of at least jf_tree_attention_workspace_size(...) bytes
 *                (may be NULL when that size is 0); contents need no initialisation.
 *   dev_err      JF_DEVERR_BAD_PAGE / _BAD_PREFIX / _TIMEOUT.  May be NULL.
 * Limits: D in {64, 128}; page_size == 16; Hq % Hkv == 0 and G = Hq / Hkv a power of
 * two <= 128; 1 <= N <= JF_MAX_NODES; max_pages * page_size >= N; q, the caches, out and
 * the workspace 16-byte aligned, mask 8-byte aligned.  Others return JF_ERR_UNSUPPORTED /
 * JF_ERR_MISALIGNED.  Every slot of the tree region must hold finite K/V values; slots past
 * P_b + N in the last page may hold anything (they are zeroed on chip before use).
 */
jf_status jf_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_table, const int32_t* prefix_len,
                            const uint64_t* mask, int32_t B, int32_t N, int32_t Hq,
                            int32_t Hkv, int32_t D, int32_t page_size, int32_t max_pages,
                            int32_t num_pages, float scale, void* out, float* lse,
                            void* workspace, size_t workspace_bytes, int32_t* dev_err,
                            jf_stream_t stream);

/*
 * Bytes of device workspace jf_tree_verify needs on the CURRENT device (per-chunk argmax
 * partials).  Returns (size_t)-1 for unsupported sizes.
 */
size_t jf_tree_verify_workspace_size(int32_t B, int32_t N, int32_t V);

/*
 * jf_tree_verify -- greedy tree verification (the target checks every drafted node in
 * one pass and keeps the longest drafted prefix it agrees with; explainer §4 counts the
 * accepted tokens tau).
 *   argmax[b][i] = smallest v with logits[b][i][v] == max_v logits[b][i][v]
 *                  (values compared as real numbers, -0 == +0; inputs must be finite)
 *   node c (c >= 1) is accepted iff draft[b][c] == argmax[b][parent[b][c]]
 *   len(i) = 0 if i has no accepted child, else 1 + max len over accepted children
 *   accept_len[b] = len(root)       (accepted draft nodes; the root is not counted)
 *   path[b]       = root, then repeatedly the accepted child with the greatest len
 *                   (ties: smallest node id); remaining entries -1
 *   bonus[b]      = argmax[b][last node of path[b]]
 *
 *   logits     [B][N][V], dtype JF_DTYPE_BF16 or JF_DTYPE_F32.
 *   draft      int32 [B][N]; draft[b][0] (the root's token) is ignored.
 *   parent     int32 [B][N].
 *   argmax     int32 [B][N] or NULL.
 *   accept_len int32 [B];  path int32 [B][N];  bonus int32 [B].
 *   workspace  at least jf_tree_verify_workspace_size(B, N, V) bytes, no initialisation.
 *   dev_err    JF_DEVERR_BAD_PARENT / _BAD_TOKEN.  May be NULL.
 * Limits: 1 <= N <= JF_MAX_NODES, 1 <= V < 2^31.
 */
jf_status jf_tree_verify(const void* logits, int32_t dtype, const int32_t* draft,
                         const int32_t* parent, int32_t B, int32_t N, int32_t V,
                         int32_t* argmax, int32_t* accept_len, int32_t* path, int32_t* bonus,
                         void* workspace, size_t workspace_bytes, int32_t* dev_err,
                         jf_stream_t stream);

/*
 * jf_tree_verify_static -- the same computation and outputs as jf_tree_verify, for
 * callers that cannot allocate device memory on their call path: for example a serving
 * engine that reserves all free device memory for its KV-cache pool at start-up, or a
 * plug-in running inside a host application that does not expose an allocator.  The
 * paper has no counterpart; this is a packaging variant of the verify call.
 *
 * Instead of a caller-provided workspace it uses a fixed scratch array compiled into the
 * library (JF_VERIFY_STATIC_SCRATCH_KEYS uint64 entries, 4 MiB), which every GPU that
 * loads the library keeps until the process exits.  The call itself allocates nothing.
 *   - The first call on each device looks up the array's device address with
 *     cudaGetSymbolAddress (a runtime query, no allocation) while that device is current,
 *     and caches it for the life of the process; make that first call before any stream
 *     capture.  The cache does not survive a reset of the device's context
 *     (cudaDeviceReset): do not use this call on a device after resetting it.
 *   - Capacity: B * N * chunks entries, where chunks = jf_tree_verify_workspace_size(B, N,
 *     V) / (8 * B * N).  Larger problems return JF_ERR_SCRATCH_CAPACITY and launch nothing.
 *   - The array is shared by every call and keeps the last call's contents; nothing in it
 *     needs to start at zero (each entry read is written earlier in the same call).
 *     Calls whose kernels overlap on the GPU (different streams, or different host
 *     threads) race on it: serialise them.
 * Arguments, limits and device error bits are those of jf_tree_verify.
 */
#define JF_VERIFY_STATIC_SCRATCH_KEYS (1u << 19)
jf_status jf_tree_verify_static(const void* logits, int32_t dtype, const int32_t* draft,
                                const int32_t* parent, int32_t B, int32_t N, int32_t V,
                                int32_t* argmax, int32_t* accept_len, int32_t* path,
                                int32_t* bonus, int32_t* dev_err, jf_stream_t stream);

/*
 * Vocabulary-sharded greedy verification.  When the target model's output layer is split
 * by vocabulary across GPUs (tensor parallelism), each GPU holds the logits of one token
 * range [vocab_offset, vocab_offset + V_shard) for every node.  The verify rule of
 * jf_tree_verify (one target pass scores every drafted node; explainer §4) needs only
 * each node's argmax, and the argmax over the whole vocabulary is the best of the
 * per-range argmaxes (greatest value, then lowest token id), so the ranges exchange one
 * 8-byte key per node and range chunk and every GPU runs the same walk on them:
 *
 *   1. chunks = jf_tree_verify_shard_chunks(B, N, largest V_shard)  (same on every GPU)
 *   2. jf_tree_verify_shard_keys(logits_shard, ..., keys_local)  keys_local [B*N][chunks]
 *   3. the caller all-gathers keys_local into keys [S][B*N][chunks] (S ranges, any
 *      order; e.g. torch.distributed.all_gather_into_tensor on uint64 / int64 storage)
 *   4. jf_tree_verify_from_keys(keys, S, chunks, ...)  -> the outputs of jf_tree_verify
 *
 * A key is (order-preserving bits of the value) << 32 | (0xFFFFFFFF - global token id):
 * the larger key (as an UNSIGNED integer) is the larger value, then the lower id; -0 and
 * +0 compare equal.  Key 0 marks a chunk with no tokens.  A signed MAX all-reduce of the
 * int64 storage would order positive values below negative ones: gather, do not reduce.
 * The library runs no collective itself.
 */

/* Chunks per node of jf_tree_verify_shard_keys for this shard size; -1 for unsupported
 * sizes.  Depends on the CURRENT device's SM count: use the same value on every GPU. */
int32_t jf_tree_verify_shard_chunks(int32_t B, int32_t N, int32_t V_shard);

/*
 * jf_tree_verify_shard_keys -- per-chunk argmax keys of one vocabulary range.
 *   logits_shard [B][N][V_shard], dtype JF_DTYPE_BF16 or JF_DTYPE_F32 (finite values).
 *   vocab_offset global id of the range's first token (>= 0; vocab_offset + V_shard < 2^31).
 *   chunks       >= 1, the same on every range: normally jf_tree_verify_shard_chunks(B, N,
 *                largest V_shard).  The range is cut into chunks slices of equal length (a
 *                multiple of 8 tokens); slices past its end get key 0.
 *   keys         uint64 [B*N][chunks], device, 8-byte aligned; fully written.
 * Launches one kernel and allocates nothing.
 * Errors: JF_ERR_INVALID_ARGUMENT (null pointer, bad dtype, B, N, V_shard or chunks < 1,
 * negative offset), JF_ERR_UNSUPPORTED (N > JF_MAX_NODES, ids past 2^31 - 1, grid too
 * large), JF_ERR_MISALIGNED.
 */
jf_status jf_tree_verify_shard_keys(const void* logits_shard, int32_t dtype, int32_t B,
                                    int32_t N, int32_t V_shard, int32_t vocab_offset,
                                    int32_t chunks, uint64_t* keys, jf_stream_t stream);

/*
 * jf_tree_verify_from_keys -- the walk of jf_tree_verify on gathered keys (fixed-size
 * trees: every sequence has N nodes).
 *   keys       uint64 [S][B*N][chunks], device: every range's jf_tree_verify_shard_keys
 *              output.  argmax[b][i] = the token id of the largest key of row b*N + i;
 *              the ranges together must cover the vocabulary [0, V).
 *   S, chunks  >= 1.
 *   draft, parent, argmax, accept_len, path, bonus, dev_err: as in jf_tree_verify
 *              (V bounds the draft tokens checked for JF_DEVERR_BAD_TOKEN).
 *   workspace  at least 8 * B * N bytes, 8-byte aligned, no initialisation.
 * Launches two kernels (the merge of the keys, then the walk) and allocates nothing.
 * Errors: JF_ERR_INVALID_ARGUMENT, JF_ERR_UNSUPPORTED (N > JF_MAX_NODES),
 * JF_ERR_WORKSPACE_TOO_SMALL, JF_ERR_MISALIGNED.
 */
jf_status jf_tree_verify_from_keys(const uint64_t* keys, int32_t S, int32_t chunks,
                                   const int32_t* draft, const int32_t* parent, int32_t B,
                                   int32_t N, int32_t V, int32_t* argmax, int32_t* accept_len,
                                   int32_t* path, int32_t* bonus, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, jf_stream_t stream);

/*
 * jf_debug_set_wait_limit_ns -- test hook for the bounded waits (no counterpart in the
 * paper).  Every wait of the tree-attention kernels on their own pipeline (a copy landing,
 * a tensor-core step finishing, a softmax pass) gives up after limit_ns nanoseconds,
 * sets JF_DEVERR_TIMEOUT in *dev_err and lets the kernel finish; the waits that drain a
 * CTA's own copies and tensor-core work before it exits keep the default limit, so an
 * abandoned call still returns with its shared memory and tensor memory released.
 * With withhold_arrivals != 0 the warps that tell the tensor-core issuer "this key tile's
 * data has landed" never do, so the issuer waits for a barrier phase nothing completes:
 * the way to make a wait run out on purpose.  (0, 0) restores normal operation (one-second
 * limit).  Applies to the CURRENT device and to calls launched after it returns (it
 * synchronises with the device); not for use while other threads launch attention calls.
 * Returns JF_ERR_CUDA if the device cannot be written.
 */
jf_status jf_debug_set_wait_limit_ns(uint64_t limit_ns, int32_t withhold_arrivals);

/*
 * jf_tree_verify_sampled -- lossless (stochastic) tree verification.  The pages call
 * draft-then-verify lossless -- the output follows the target model's distribution
 * (qxai.app commentary, "まず、何が問題なのか" and "慎重に見るべき点"; explainer §1) --
 * without giving the rule; this call uses the multi-step speculative sampling of SpecInfer
 * (Miao et al., ASPLOS 2024) for deterministic drafts, whose children are fixed candidate
 * tokens (point-mass draft distributions):
 *   p_u = softmax(logits[b][u] / temperature) at node u, starting at the root;
 *   the children c of u are tested in increasing node id: with R the probability mass of
 *   p_u left after removing the tokens rejected so far at u, c (token x = draft[b][c]) is
 *   accepted iff uniform[b][c] * R < p_u(x) with x not yet removed; on acceptance the walk
 *   continues at c, on rejection x is removed;
 *   when no child of u is accepted (or u has none), bonus[b] = the smallest token y whose
 *   cumulative residual probability exceeds bonus_uniform[b] * R.
 *   accept_len[b] = accepted nodes; path[b] = root, then the accepted nodes, -1 padded.
 * Every emitted token (accepted drafts, then the bonus) is then a sample of the target's
 * distribution at its position.
 *   logits         [B][N][V] bf16 or fp32 (dtype), finite.
 *   uniform        float [B][N] in [0, 1): the number drawn when node c is tested (entry
 *                  0 unused; each node is tested at most once).
 *   bonus_uniform  float [B] in [0, 1).
 *   temperature    > 0.
 *   workspace      at least jf_tree_verify_workspace_size(B, N, V) bytes, no initialisation.
 *   dev_err        JF_DEVERR_BAD_PARENT / _BAD_TOKEN.  May be NULL.
 * Precision: p is computed in fp64 from per-chunk fp32 maxima and Kahan-compensated fp32
 * sums of exponentials (relative error about 1e-6), so a decision whose threshold lies
 * closer than that to its boundary may differ from an exact computation.
 * Limits: 1 <= N <= JF_MAX_NODES, 1 <= V < 2^31.
 */
jf_status jf_tree_verify_sampled(const void* logits, int32_t dtype, const int32_t* draft,
                                 const int32_t* parent, const float* uniform,
                                 const float* bonus_uniform, float temperature, int32_t B,
                                 int32_t N, int32_t V, int32_t* accept_len, int32_t* path,
                                 int32_t* bonus, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_err, jf_stream_t stream);

/* ---------------------------------------------------------------- ragged trees
 * One batch may mix tree budgets: the best budget depends on the serving load (explainer
 * §4, serving performance), so sequences of one step can carry trees of different sizes.
 * The three calls below are jf_build_tree_mask, jf_tree_attention and jf_tree_verify with
 * one more argument, tree_len int32 [B] (device): sequence b's tree has the nodes
 * 0 .. n_b - 1, n_b = tree_len[b], 1 <= n_b <= N; arrays keep their [B][N] shapes and
 * entries of nodes i >= n_b are padding.  With tree_len[b] == N for every b each call
 * computes what its fixed-size counterpart computes (the attention call up to
 * floating-point summation order, since a ragged call never takes the stream-K dispatch,
 * whose ranges cannot skip padding row groups).  A tree_len entry outside
 * [1, N] sets JF_DEVERR_BAD_TREE_LEN and is clamped into that range.
 *   jf_build_tree_mask_ragged: parent[b][i] is read for i < n_b only; rows i >= n_b get
 *     all-zero mask words and depth = pos = -1.
 *   jf_tree_attention_ragged: the tree's keys/values are the n_b positions
 *     P_b .. P_b + n_b - 1; block-table entries past ceil((P_b + n_b) / page_size) are
 *     never read and K/V slots past P_b + n_b may hold anything (the padding nodes need no
 *     K/V at all).  Rows i < n_b are as in jf_tree_attention; rows i >= n_b of out and lse
 *     carry no meaning (they may be left unwritten or hold anything).  Groups of 128-256
 *     query rows that hold only padding nodes are not computed, so a batch of small trees
 *     costs about what its trees need.
 *   jf_tree_verify_ragged: nodes i >= n_b are never accepted and their parent and draft
 *     entries are not read; argmax is still written for every row, so logits rows
 *     i >= n_b must be readable (their values do not matter).  path[b] lists nodes < n_b.
 * Workspace sizes: jf_tree_attention_workspace_size and jf_tree_verify_workspace_size
 * with the same N.
 */
jf_status jf_build_tree_mask_ragged(const int32_t* parent, const int32_t* prefix_len,
                                    const int32_t* tree_len, int32_t B, int32_t N,
                                    uint64_t* mask, int32_t* depth, int32_t* pos,
                                    int32_t* dev_err, jf_stream_t stream);
jf_status jf_tree_attention_ragged(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* prefix_len,
                                   const int32_t* tree_len, const uint64_t* mask, int32_t B,
                                   int32_t N, int32_t Hq, int32_t Hkv, int32_t D,
                                   int32_t page_size, int32_t max_pages, int32_t num_pages,
                                   float scale, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, jf_stream_t stream);
jf_status jf_tree_verify_ragged(const void* logits, int32_t dtype, const int32_t* draft,
                                const int32_t* parent, const int32_t* tree_len, int32_t B,
                                int32_t N, int32_t V, int32_t* argmax, int32_t* accept_len,
                                int32_t* path, int32_t* bonus, void* workspace,
                                size_t workspace_bytes, int32_t* dev_err, jf_stream_t stream);

/*
 * Packed (cu_seqlens) layout of ragged trees: the per-node arrays hold only real nodes,
 * sequence after sequence.  cu_seqlens int32 [B + 1] (device) with cu_seqlens[0] = 0 and
 * cu_seqlens[B] = T: sequence b's n_b = cu_seqlens[b + 1] - cu_seqlens[b] nodes
 * (1 <= n_b <= N_max) sit at rows cu_seqlens[b] .. cu_seqlens[b + 1] - 1, and parent and
 * path entries are node ids within the sequence (0 .. n_b - 1).  Each call computes, for
 * every sequence, what its _ragged counterpart computes with N = N_max and
 * tree_len[b] = n_b (same kernels, same plan: outputs equal bit for bit), with packed
 * arrays in place of padded ones:
 *   parent, draft, depth, pos, argmax   int32 [T]
 *   mask                                uint64 [T][W], W = ceil(N_max / 64)
 *   q, out                              bf16 [T][Hq][D]
 *   lse                                 fp32 [Hq][T]
 *   logits                              [T][V]
 *   accept_len, bonus [B] and path [B][N_max] keep their shapes.
 * A span that is empty, longer than N_max, decreasing or outside [0, T) sets
 * JF_DEVERR_BAD_TREE_LEN; nothing of that sequence is then read or written except its
 * accept_len (0), path (0, then -1) and bonus (-1) in verify.  T is a host argument
 * (the caller knows the batch it packed).  Workspaces: jf_tree_attention_workspace_size
 * with N = N_max; jf_tree_verify_packed_workspace_size(T, V) for verify.
 * Limits: as the padded calls, plus 1 <= T and T + N_max < 2^31.
 */
jf_status jf_build_tree_mask_packed(const int32_t* parent, const int32_t* prefix_len,
                                    const int32_t* cu_seqlens, int32_t B, int32_t N_max,
                                    int32_t T, uint64_t* mask, int32_t* depth, int32_t* pos,
                                    int32_t* dev_err, jf_stream_t stream);
jf_status jf_tree_attention_packed(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* prefix_len,
                                   const int32_t* cu_seqlens, const uint64_t* mask, int32_t B,
                                   int32_t N_max, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                   int32_t page_size, int32_t max_pages, int32_t num_pages,
                                   float scale, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, jf_stream_t stream);
size_t jf_tree_verify_packed_workspace_size(int32_t T, int32_t V);
jf_status jf_tree_verify_packed(const void* logits, int32_t dtype, const int32_t* draft,
                                const int32_t* parent, const int32_t* cu_seqlens, int32_t B,
                                int32_t N_max, int32_t T, int32_t V, int32_t* argmax,
                                int32_t* accept_len, int32_t* path, int32_t* bonus,
                                void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                jf_stream_t stream);

/*
 * Lossless verification of ragged trees: jf_tree_verify_sampled with per-sequence tree
 * sizes, padded (tree_len [B], as the _ragged calls) or packed (cu_seqlens [B + 1], as the
 * _packed calls; uniform then float32 [T], one draw per packed node).  Padding nodes are
 * never read and never accepted; every sequence's accept_len, path and bonus are what
 * jf_tree_verify_sampled gives on the sequence's first n_b nodes alone, with the same
 * random numbers.  Workspace: jf_tree_verify_workspace_size(B, N, V) for the ragged call,
 * jf_tree_verify_packed_workspace_size(T, V) for the packed one.  A tree_len entry outside
 * [1, N] is reported and clamped; a bad packed span is reported and its sequence gets
 * accept_len 0, path (0, then -1) and bonus -1 without any of its rows being read.
 */
jf_status jf_tree_verify_sampled_ragged(const void* logits, int32_t dtype, const int32_t* draft,
                                        const int32_t* parent, const int32_t* tree_len,
                                        const float* uniform, const float* bonus_uniform,
                                        float temperature, int32_t B, int32_t N, int32_t V,
                                        int32_t* accept_len, int32_t* path, int32_t* bonus,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* dev_err, jf_stream_t stream);
jf_status jf_tree_verify_sampled_packed(const void* logits, int32_t dtype, const int32_t* draft,
                                        const int32_t* parent, const int32_t* cu_seqlens,
                                        const float* uniform, const float* bonus_uniform,
                                        float temperature, int32_t B, int32_t N_max, int32_t T,
                                        int32_t V, int32_t* accept_len, int32_t* path,
                                        int32_t* bonus, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_err, jf_stream_t stream);

/* ---------------------------------------------------------------- before verification
 * jf_build_draft_tree -- builds the draft tree from per-depth draft logits.  JetFlow
 * explainer ("JetFlow: Breaking the Scaling Ceiling of Speculative Decoding with Parallel
 * Tree Drafting"), technical summary §2 "Method", tree construction: the draft head emits
 * logits for every depth in one pass, a branch score (by default the cumulative draft
 * log-probability) ranks nodes, and a best-first expansion builds the tree up to a budget.
 * Computed here (the pages fix no more detail; this is the plainest reading):
 *   1. candidates: for sequence b and depth d = 1..Dmax (row d-1 of draft_logits[b]), the
 *      K tokens with the largest logits (lower token id on ties), in that order, with
 *      log-probabilities logit - logsumexp(row), fp32 -> cand_token / cand_logp
 *      [B][Dmax][K].
 *   2. tree: the root (depth 0, score 0, token root_token[b]) and, below every node of
 *      depth d < Dmax, the K depth-(d+1) candidates as children (child score =
 *      fp32(parent score + candidate log-prob)).  Best-first expansion to N nodes takes
 *      nodes in the order (score descending, depth ascending, rank path ascending); node
 *      ids follow that order, so parent[i] < i.  Outputs parent (root -1), draft (token;
 *      root_token[b] or -1 for the root when root_token is NULL), depth and score (may be
 *      NULL), all [B][N].
 * Arguments: draft_logits bf16 or fp32 [B][Dmax][V] (dtype JF_DTYPE_*), device pointers.
 * Limits: 1 <= K <= 8, 1 <= Dmax <= 16, 1 <= N <= 256, V >= K, and
 *   the candidate lattice must hold N nodes (1 + K + ... + K^Dmax >= N); otherwise
 *   JF_ERR_UNSUPPORTED.  Logits must be finite.
 */
jf_status jf_build_draft_tree(const void* draft_logits, int32_t dtype, const int32_t* root_token,
                              int32_t B, int32_t Dmax, int32_t V, int32_t K, int32_t N,
                              int32_t* cand_token, float* cand_logp, int32_t* parent,
                              int32_t* draft, int32_t* depth, float* score, jf_stream_t stream);

/*
 * jf_build_draft_tree_ragged -- the same with a budget per sequence (the best budget depends
 * on the load, explainer §4): budget int32 [B] (device), each clamped to [1, N]
 * (JF_DEVERR_BAD_TREE_LEN in *dev_err, which may be NULL, when one is outside).  Sequence
 * b's tree is the best-first tree of budget[b] nodes, nodes 0 .. budget[b] - 1 of the
 * [B][N] outputs (equal to what jf_build_draft_tree gives with N = budget[b]); the
 * remaining entries are padding (parent = draft = depth = -1, score = -inf), so budget
 * serves as tree_len for the _ragged calls.  Limits as jf_build_draft_tree.
 */
jf_status jf_build_draft_tree_ragged(const void* draft_logits, int32_t dtype,
                                     const int32_t* root_token, const int32_t* budget, int32_t B,
                                     int32_t Dmax, int32_t V, int32_t K, int32_t N,
                                     int32_t* cand_token, float* cand_logp, int32_t* parent,
                                     int32_t* draft, int32_t* depth, float* score,
                                     int32_t* dev_err, jf_stream_t stream);

/* ---------------------------------------------------------------- after verification
 * jf_compact_accepted_kv -- moves the K/V of the accepted draft path next to the prefix,
 * so the next decoding step continues from one contiguous context.  JetFlow explainer
 * ("JetFlow: Breaking the Scaling Ceiling of Speculative Decoding with Parallel Tree
 * Drafting"), technical summary §2 "Method": draft-tree nodes keep their K/V after the
 * prefix and the accepted branch is what the target continues from; the pages do not
 * spell out the cache update, so the plainest reading is implemented:
 *   for every sequence b with a = accept_len[b] and P = prefix_len[b], for k = 1..a in
 *   increasing order, the K and V rows (all kv-heads) at logical position P + path[b][k]
 *   are copied to position P + k; then new_prefix_len[b] = P + a + 1 (the root and the
 *   accepted nodes join the prefix; the bonus token's K/V come from the next forward
 *   pass).  Because path[k] >= k rises strictly, a source is never overwritten before
 *   it is read in that order; the kernel reproduces exactly this sequential result.
 * Arguments:
 *   k_cache, v_cache  bf16 [num_pages][page_size][Hkv][D], modified in place.
 *   block_table       int32 [B][max_pages]; prefix_len int32 [B] (read only).
 *   path, accept_len  int32 [B][N] and [B], as written by jf_tree_verify.
 *   new_prefix_len    int32 [B] out; must not alias prefix_len.
 *   dev_err           may be NULL.
 * Only positions P + 1 .. P + a are written.  A sequence whose prefix length, accepted
 * length, path (path[0] == 0, strictly increasing, inside [0, N)) or block-table entries
 * are malformed is left unchanged (new_prefix_len = P) and sets JF_DEVERR_BAD_PREFIX,
 * JF_DEVERR_BAD_PATH or JF_DEVERR_BAD_PAGE.
 * Limits: D in {64, 128}, page_size 16, 1 <= N <= JF_MAX_NODES, caches 16-byte aligned.
 */
jf_status jf_compact_accepted_kv(void* k_cache, void* v_cache, const int32_t* block_table,
                                 const int32_t* prefix_len, const int32_t* path,
                                 const int32_t* accept_len, int32_t B, int32_t N, int32_t Hkv,
                                 int32_t D, int32_t page_size, int32_t max_pages,
                                 int32_t num_pages, int32_t* new_prefix_len, int32_t* dev_err,
                                 jf_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* JF_H_ */
