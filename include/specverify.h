/*
 * specverify.h - C ABI of libspecverify, the batched verify step of
 * speculative decoding on one GPU (sm_103a).
 *
 * The verify step takes, for each of B sequences, the target model's
 * distribution at the K draft positions plus one more after the last draft
 * (K+1 rows of V logits), the draft model's K rows and the K draft tokens,
 * checks the drafts left to right, and commits the accepted drafts followed
 * by one target token (a correction at the first rejection, or a bonus token
 * when every draft is accepted). Sources:
 *   "Inference-4" (brunomaga.github.io), section "Draft-model speculative
 *     decoding": the K+1 rows, the greedy rule (accept while the draft equals
 *     the target's most likely token; correction or bonus from the target),
 *     the sampling rule (accept x with probability min(1, P_t(x)/P_d(x)); on
 *     rejection draw from the normalised residual max(0, P_t - P_d)), and the
 *     note that sequences of a batch accept different numbers of tokens.
 *   "Speculative decoding" (leoniemonigatti.com blog), section "Rejection
 *     sampling": the same rule and the bonus token when all drafts pass.
 *   "Speculative decoding" (denimpatel.github.io interactive course), section
 *     "Memory-bound, not compute-bound": verification is a forward pass whose
 *     query dimension is K (+1), the target's LM head included, which the
 *     fused entry point spec_verify_lmhead covers.
 *
 * Conventions shared by every entry point:
 *   - All array arguments are DEVICE pointers to caller-owned memory on the
 *     current CUDA device; the library allocates nothing and frees nothing.
 *   - Layouts are dense row-major: logits [B, K+1, V] and [B, K, V] with V
 *     innermost; each row must start on a multiple of its element size.
 *   - Calls are asynchronous and stream-ordered on `stream` (NULL = the
 *     legacy default stream); no call synchronises the host. Buffers must
 *     stay valid until the work on `stream` completes.
 *   - Host-detectable errors return a status before anything is launched and
 *     leave the outputs untouched. A failed launch returns SV_ERR_CUDA.
 *   - Device-detectable errors never trap: a sequence whose draft token is
 *     outside [0, V), or whose rows contain no finite maximum (all -inf, or a
 *     NaN or +inf), gets n_accepted = -1 and every token -1, and the bits of
 *     sv_device_flag are OR-ed into the optional status word.
 *   - Temperature: both distributions are softmax(logits / T). Greedy mode
 *     ignores T. -inf logits are allowed and mean probability zero.
 *   - Random numbers: Philox4x32-10 (Salmon et al., SC'11) with counter
 *     (pos, seq_lo, seq_hi, 0) and key (seed_lo, seed_hi); word 0 gives the
 *     accept uniform u of draft position pos, word 1 the uniform u2 of the
 *     residual or bonus draw at that position; each is (w >> 8) * 2^-24. A
 *     draft x at position i is accepted iff u * P_d(x) < P_t(x).
 *   - The draw is the inverse CDF in index order: the smallest token k whose
 *     cumulative mass exceeds u2 times the total mass.
 *   - The thread-safety of a call is that of its stream: concurrent calls on
 *     different streams with disjoint outputs are safe.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* sv_stream_t;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;
typedef enum { SV_GREEDY = 0, SV_SAMPLE = 1 } sv_mode;

typedef enum {
    SV_OK = 0,
    SV_ERR_NULL = 1,          /* a required pointer is NULL                     */
    SV_ERR_SHAPE = 2,         /* B < 1, K outside [1, 31], V < 2, d bad, ...    */
    SV_ERR_DTYPE = 3,         /* unknown dtype                                  */
    SV_ERR_TEMPERATURE = 4,   /* sample mode with T not finite or T <= 0        */
    SV_ERR_WORKSPACE = 5,     /* workspace NULL or smaller than required        */
    SV_ERR_ARCH = 6,          /* the current device is not compute capability 10.3 */
    SV_ERR_CUDA = 7,          /* a CUDA runtime call or launch failed           */
    SV_ERR_MODE = 8,          /* unknown mode                                   */
    SV_ERR_ALIGN = 9,         /* a pointer is not aligned to its element size   */
    SV_ERR_CONFIG = 10,       /* a requested launch parameter cannot be used    */
    SV_ERR_NOT_IMPLEMENTED = 11,
    SV_ERR_SCRATCH_LIMIT = 12 /* needs more than SV_LMHEAD_SCRATCH_BYTES     */
} sv_status;

/* Bits OR-ed into the optional device status word. */
typedef enum {
    SV_FLAG_BAD_TOKEN = 1u,        /* a draft token outside [0, V)                 */
    SV_FLAG_BAD_ROW = 2u,          /* a row with no finite maximum                 */
    SV_FLAG_RESIDUAL_FALLBACK = 4u,/* a residual summed to 0 in float; P_t used    */
    SV_FLAG_DRAW_EDGE = 8u,        /* a draw landed past the summed mass (rounding)*/
    SV_FLAG_BAD_MODE = 16u,        /* a per-sequence mode that is neither greedy nor
                                      sample, or sample mode without draft logits  */
    SV_FLAG_TIMEOUT = 32u,         /* a bounded wait inside the kernel gave up; the
                                      sequence is reported invalid                 */
    SV_FLAG_BAD_LENGTH = 64u,      /* a per-sequence draft length outside [0, K]   */
    SV_FLAG_BAD_TREE = 128u,       /* a tree node whose parent is not an earlier
                                      node                                         */
    SV_FLAG_DEBUG_BOUNDS = 256u    /* debug builds only (libspecverify_debug.so,
                                      compiled with SPECVERIFY_DEBUG): the verify
                                      kernel was about to access global memory
                                      outside every buffer of the call; it skipped
                                      that access instead                          */
} sv_device_flag;

/* Batched verify over logits already in device memory.
 *   target_logits  [B, K+1, V] of `dtype` (device): the target's rows at the K
 *                  draft positions and after the last draft.
 *   draft_logits   [B, K, V] of `dtype` (device): the draft's rows; may be
 *                  NULL in greedy mode (never read there).
 *   draft_tokens   [B, K] int32 (device): the drafts x_0..x_{K-1}.
 *   B >= 1, 1 <= K <= 31, V >= 2; dtype SV_F32 or SV_BF16.
 *   temperature    T of both softmaxes in sample mode (finite, > 0).
 *   mode           SV_GREEDY or SV_SAMPLE for the whole batch.
 *   seed           Philox key; the sequence id of row b is b.
 *   out_tokens     [B, K+1] int32 (device): x_0..x_{j-1}, then the correction
 *                  or bonus token, then -1 padding.
 *   out_n_accepted [B] int32 (device): j, the number of accepted drafts
 *                  (0..K), or -1 for an invalid sequence.
 * Returns SV_OK once the work is enqueued. */
sv_status spec_verify(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, int B, int K, int V,
                      sv_dtype dtype, float temperature, sv_mode mode,
                      uint64_t seed, int32_t* out_tokens,
                      int32_t* out_n_accepted, sv_stream_t stream);

/* Arguments of spec_verify_ex. Zero-initialise, then fill what is used. */
typedef struct {
    const void* target_logits;   /* [B, K+1, V] dtype (device)                    */
    const void* draft_logits;    /* [B, K, V] dtype (device); NULL if all greedy  */
    const int32_t* draft_tokens; /* [B, K] int32 (device)                         */
    int B, K, V;
    sv_dtype dtype;
    float temperature;
    sv_mode mode;                /* the mode of every sequence when modes == NULL */
    const int32_t* modes;        /* [B] int32 (device) per-sequence SV_GREEDY or
                                    SV_SAMPLE, or NULL; other values make the
                                    sequence invalid                               */
    uint64_t seed;
    const uint64_t* seq_ids;     /* [B] uint64 (device) Philox sequence ids, or
                                    NULL (id = b); lets a batch split across calls
                                    keep each sequence's random stream            */
    int32_t* out_tokens;         /* [B, K+1] int32 (device)                       */
    int32_t* out_n_accepted;     /* [B] int32 (device)                            */
    float* out_p_target;         /* [B, K] float (device) or NULL: P_t(x_i) at the
                                    call's temperature (NaN for greedy sequences) */
    float* out_p_draft;          /* [B, K] float (device) or NULL: P_d(x_i)       */
    float* out_residual_mass;    /* [B] float (device) or NULL: total mass of the
                                    final draw (residual after a rejection, P_t of
                                    row K for the bonus); NaN when greedy         */
    uint32_t* status_word;       /* device uint32 or NULL: sv_device_flag bits are
                                    OR-ed in; never cleared by the library        */
    int cluster_size;            /* CTAs that share one sequence: 0 = automatic,
                                    else 1, 2, 4, 8 or 16                         */
    sv_stream_t stream;
    uint32_t flags;              /* SV_ARG_* bits, 0 for none                     */
    const int32_t* draft_lens;   /* [B] int32 (device) or NULL: sequence b verifies
                                    only its first draft_lens[b] drafts (0..K;
                                    continuous batching). It reads target rows
                                    0..Kb and draft rows 0..Kb-1 of its block and
                                    writes -1 / NaN past Kb; a value outside
                                    [0, K] makes the sequence invalid            */
    float* out_draw_edges;       /* [B, 2] float (device) or NULL: for a sample
                                    sequence, the distances from the final draw's
                                    target t = u2 * (total mass) down to the lower
                                    and up to the upper edge of the chosen token's
                                    cumulative interval, in probability units, as
                                    the kernel computed them (0, 0 when rounding
                                    left t at or past the total); NaN for greedy
                                    or invalid sequences                          */
    int seqs_per_cluster;        /* calls without SV_ARG_OVERLAP_PREVIOUS only:
                                    0 = automatic; 1 = one cluster per sequence;
                                    2..8 = clusters of cluster_size CTAs (8 when
                                    cluster_size is 0) that each verify up to
                                    this many sequences, every CTA streaming its
                                    slice of V of all of them, so that a large
                                    batch spreads evenly over the SMs (B <= 256,
                                    at most 120 rows read per cluster, each of
                                    its drawing sequences keeping at least
                                    cluster_size / seqs_per_cluster CTAs;
                                    otherwise SV_ERR_CONFIG). Automatic groups
                                    a batch of at least 19 sequences when such a
                                    plan fills about two CTAs per SM and
                                    cluster_size is 0                              */
} sv_verify_args;

/* sv_verify_args.flags: the inputs of this call are not written by the work
 * enqueued just before it on `stream`, so the call may start reading them
 * while that work (typically the previous verify call) is still running. Its
 * outputs are still written only after that work has completed. Without the
 * flag a call starts after everything before it on the stream. Such a call
 * runs one CTA per sequence (unless cluster_size asks otherwise), two per SM,
 * so that consecutive calls share the GPU; a lone call without the flag
 * spreads each sequence over a cluster of CTAs instead. */
#define SV_ARG_OVERLAP_PREVIOUS 1u

/* sv_verify_args.flags, for tests of the failure path only: every CTA also
 * waits, with a short bound, on a barrier that nothing completes. The wait
 * gives up as a real stalled copy would, and the call reports
 * SV_FLAG_TIMEOUT and marks every sequence invalid, without faulting. */
#define SV_ARG_TEST_WAIT_TIMEOUT 0x80000000u

/* sv_verify_args.flags, for tests of the debug build only: its bounds checks
 * take the target logits to end halfway through the buffer, so that every
 * access of the upper half counts as out of bounds (and is skipped, setting
 * SV_FLAG_DEBUG_BOUNDS). No access leaves the real buffer. Release builds
 * ignore the flag. */
#define SV_ARG_TEST_DEBUG_SHRINK 0x40000000u

/* spec_verify with per-sequence modes, explicit sequence ids and optional
 * probability outputs. Same conventions and errors as spec_verify. */
sv_status spec_verify_ex(const sv_verify_args* args);

/* The launch spec_verify_ex would make for these arguments. */
typedef struct {
    int grouped;              /* 1: several sequences per cluster (each CTA
                                 streams its slice of V of all of them);
                                 0: one cluster per sequence               */
    int clusters;             /* clusters in the grid                       */
    int cluster_size;         /* CTAs per cluster                           */
    int max_seqs_per_cluster; /* 1 unless grouped                           */
} sv_verify_plan;

/* Validates args exactly as spec_verify_ex does (same status on error) and
 * fills *plan with the launch it would make; reads no device memory and
 * enqueues nothing (it queries the current device's properties). */
sv_status spec_verify_plan(const sv_verify_args* args, sv_verify_plan* plan);

/* Bytes of device workspace spec_verify_lmhead needs for these sizes:
 * the fp32 logits B*(K+1)*V*4, then 8 bytes per target row and 128-column
 * tile of V (ceil(V/128)*B*(K+1)*8), then 8 bytes per draft row and tile
 * (ceil(V/128)*B*K*8), each part rounded up to 256 bytes. */
size_t spec_verify_lmhead_workspace_bytes(int B, int K, int d, int V);

/* Fused LM head + verify: the target rows are computed on the GPU as
 * logits[B*(K+1), V] = hidden[B*(K+1), d] . W[d, V] (bf16 inputs, fp32
 * accumulation on the tensor cores) and verified against the draft rows as
 * spec_verify does. ("Speculative decoding", denimpatel.github.io
 * interactive course, section "Memory-bound, not compute-bound": the K+1
 * verification rows come from one forward pass that reads the head's
 * weights once.) The GEMM's epilogue reduces every row over the 128-column
 * tiles each of its CTAs computes to a softmax partial (sample) or its
 * maximum and lowest index (greedy); the verify step merges those instead of
 * re-reading the rows and reads one target row per sequence again only for
 * the final draw. In sample mode the GEMM kernel also reduces the draft rows
 * the same way. Two kernels on `stream`; the second may start while the
 * first finishes.
 *   hidden [B, K+1, d] bf16 (device), W [d, V] bf16 (device, V contiguous),
 *   draft_logits [B, K, V] of draft_dtype (device; NULL in greedy mode),
 *   d a positive multiple of 64, V a positive multiple of 8, B * (K+1) <= 256;
 *   hidden and W 16-byte aligned. Greedy mode ignores draft_dtype.
 *   workspace: device buffer of at least
 *   spec_verify_lmhead_workspace_bytes(B, K, d, V) bytes, 256-byte aligned;
 *   its first part holds the fp32 target logits [B*(K+1), V] (sample mode
 *   only: a greedy call decides from the partials and leaves that part as
 *   it was), then the target rows' partials (one per row and GEMM CTA, room
 *   for ceil(V/128) CTAs) and (sample mode) the draft rows', 8 bytes each
 *   (every byte the call reads there it wrote first, so no initial contents
 *   are needed); it may be reused once the call's work on `stream` has
 *   completed. The size does not depend on the mode.
 * Other arguments as in spec_verify. */
sv_status spec_verify_lmhead(const void* hidden, const void* W,
                             const void* draft_logits,
                             const int32_t* draft_tokens, int B, int K, int d,
                             int V, sv_dtype draft_dtype, float temperature,
                             sv_mode mode, uint64_t seed, void* workspace,
                             size_t workspace_bytes, int32_t* out_tokens,
                             int32_t* out_n_accepted, sv_stream_t stream);

/* Greedy tree verification ("Inference-4", section "Medusa": the candidate
 * continuations of a drafter form a tree, all of them are verified in one
 * forward pass, and the longest accepted path is kept). Node 0 of each
 * sequence's tree is its root (the last committed token); node i > 0 carries
 * a candidate token and a parent node earlier than i. A node is accepted when
 * its parent is and its token is the argmax of its parent's target row; the
 * kept path ends at the deepest accepted node (lowest index among equally
 * deep ones) and is followed by the argmax of that node's row.
 *   target_logits [B, N, V] dtype (device): row i is the target's
 *     distribution after the prefix ending at node i.
 *   tree_tokens [B, N] int32 (device): node tokens (node 0's is ignored).
 *   tree_parents [B, N] int32 (device): parent of node i (node 0's ignored);
 *     a parent outside [0, i) makes the sequence invalid (SV_FLAG_BAD_TREE).
 *   1 <= N <= 32, V >= 2.
 *   out_tokens [B, N] int32 (device): the path's tokens, the next token, -1.
 *   out_n_accepted [B] int32 (device): the path length (tree nodes kept),
 *     -1 for an invalid sequence.
 *   out_last_node [B] int32 (device) or NULL: the kept path's last node (the
 *     caller keeps that node's cache entries), -1 when invalid.
 * Same stream, ownership and error conventions as spec_verify. */
sv_status spec_verify_tree(const void* target_logits, sv_dtype dtype,
                           const int32_t* tree_tokens,
                           const int32_t* tree_parents, int B, int N, int V,
                           int32_t* out_tokens, int32_t* out_n_accepted,
                           int32_t* out_last_node, sv_stream_t stream);

/* Prompt lookup drafting ("Inference-4", section "Prompt lookup decoding"):
 * for each sequence, the drafts are the tokens that followed the most recent
 * earlier occurrence of its last n-gram, trying n = max_ngram first and then
 * shorter n-grams; no drafts when none of them occurred before.
 *   tokens [B, L_max] int32 (device): each sequence's prompt and generated
 *     text so far, in its first lengths[b] entries.
 *   lengths [B] int32 (device): a length outside [0, L_max] gives -1 drafts.
 *   1 <= B <= 2^28, 1 <= max_ngram <= 16, 1 <= n_drafts <= 64 (else SV_ERR_SHAPE).
 *   out_drafts [B, n_drafts] int32 (device): the drafts, -1 padded.
 *   out_n_drafts [B] int32 (device): how many drafts (0..n_drafts; fewer when
 *     the occurrence lies near the end of the sequence).
 * Same stream, ownership and error conventions as spec_verify. */
sv_status spec_prompt_lookup(const int32_t* tokens, const int32_t* lengths,
                             int B, int L_max, int max_ngram, int n_drafts,
                             int32_t* out_drafts, int32_t* out_n_drafts,
                             sv_stream_t stream);

/* Commit step of a decode loop (the pages' loop keeps the accepted drafts and
 * the token after them): sequence b appends out_tokens[b, 0..n] (n =
 * n_accepted[b]) to its context tokens[b, lengths[b]..] and advances
 * lengths[b], stopping at L_max. An invalid verify result (n < 0 or n > K) or
 * a length outside [0, L_max] commits nothing (out_n_committed -1). The pages
 * have no such helper as a separate step; it keeps a drafting + verify loop
 * on the device (prompt lookup reads the contexts it writes).
 *   tokens [B, L_max], lengths [B] int32 (device, updated in place);
 *   out_tokens [B, K+1], n_accepted [B] int32 (device, a verify call's output);
 *   0 <= K <= 31; out_n_committed [B] int32 (device) or NULL. */
sv_status spec_commit(int32_t* tokens, int32_t* lengths, int B, int L_max,
                      const int32_t* out_tokens, const int32_t* n_accepted, int K,
                      int32_t* out_n_committed, sv_stream_t stream);

/* Capacity of the library's own device scratch used by
 * spec_verify_lmhead_noalloc: 32 MiB, i.e.
 * spec_verify_lmhead_workspace_bytes(B, K, d, V) <= 33554432 (the fp32
 * target logits and the per-tile partials; at V = 128256 that allows
 * B <= 15 for K = 3, B <= 12 for K = 4, B <= 10 for K = 5). */
#define SV_LMHEAD_SCRATCH_BYTES (32u << 20)

/* spec_verify_lmhead without a workspace argument: it allocates nothing.
 * The pages describe no such variant; it exists for callers that cannot
 * allocate device memory when they verify (a C host runtime linked without
 * an allocator of its own, or a serving loop that must not call cudaMalloc
 * or cudaFree between steps, since either may synchronise the whole device).
 * The workspace (target logits and partials) is one fixed scratch array
 * that the library's device image holds (SV_LMHEAD_SCRATCH_BYTES, 256-byte
 * aligned, one copy per device); its address is looked up once per device
 * with that device current.
 *   Arguments as in spec_verify_lmhead, minus the workspace.
 *   Nothing in the scratch needs to start at zero: the call writes every
 *   byte it reads there before reading it.
 *   Sizes whose workspace would exceed SV_LMHEAD_SCRATCH_BYTES return
 *   SV_ERR_SCRATCH_LIMIT before any work is enqueued. The limit is the
 *   mode-independent spec_verify_lmhead_workspace_bytes(B, K, d, V), which
 *   counts room for the draft rows' partials even in greedy mode.
 *   All calls on one device share the one scratch array: calls whose work
 *   may overlap (other streams, other host threads, another call before this
 *   one's work on `stream` has completed unless both are on the same stream)
 *   race on it and corrupt each other's results. Order them.
 *   The first call on each device may load the library's device image to
 *   look the address up; make that first call outside any stream capture. */
sv_status spec_verify_lmhead_noalloc(const void* hidden, const void* W,
                                     const void* draft_logits,
                                     const int32_t* draft_tokens, int B, int K,
                                     int d, int V, sv_dtype draft_dtype,
                                     float temperature, sv_mode mode,
                                     uint64_t seed, int32_t* out_tokens,
                                     int32_t* out_n_accepted,
                                     sv_stream_t stream);

/* The LM head alone: logits[M, V] = hidden[M, d] . W[d, V] with bf16 inputs
 * and fp32 accumulation on the tensor cores (the first half of
 * spec_verify_lmhead, exposed for callers that verify in a separate step).
 *   hidden [M, d] bf16 (device, d contiguous), W [d, V] bf16 (device, V
 *   contiguous), out [M, V] fp32 (device). 1 <= M <= 256, d a positive
 *   multiple of 64, V a positive multiple of 8; hidden and W 16-byte aligned. */
sv_status spec_lmhead_logits(const void* hidden, const void* W, int M, int d, int V, float* out,
                             sv_stream_t stream);

/* Static description of a status code (never NULL). */
const char* sv_status_string(sv_status status);

/* The CUDA error behind the last SV_ERR_CUDA on this host thread (0 if none). */
int sv_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int sv_version(void);

/* sizeof(sv_verify_args) as compiled into the library, so that bindings can
 * check their copy of the struct layout. */
size_t sv_verify_args_size(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
