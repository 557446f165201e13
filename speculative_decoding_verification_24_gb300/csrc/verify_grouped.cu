// Verify kernel for one call alone over a large batch: several sequences per
// cluster, every CTA of the cluster streaming its slice of V of all of them.
//
// It applies the rules verify_logits_kernel applies ("Inference-4"
// (brunomaga.github.io), section "Draft-model speculative decoding";
// "Speculative decoding" (leoniemonigatti.com blog), section "Rejection
// sampling") with the same arithmetic: the same float32 chunk reductions,
// merges, accept test and float-float draw. Its partials combine the chunks
// in another order (a warp takes a contiguous run of chunks, a draw's row is
// split over fewer CTAs), so its float statistics can differ from the other
// kernel's in the last bits; both are checked against the oracle.
//
// Why a second kernel: with one cluster per sequence a lone call places
// B * CS CTAs on the SMs, and unless that fills every SM evenly (two CTAs per
// SM) some SMs stream twice the bytes of others and set the call's time
// (256 sequences on 152 SMs: 104 SMs with two). Here n_cl clusters of CS CTAs
// (n_cl * CS close to two per SM) each take about B / n_cl sequences, so
// every CTA streams about the same bytes.
//
// Layout of the work (one launch, no global scratch):
//   assign  Every CTA orders the batch by rows read (2 Kb + 1 for a sample
//           sequence, Kb + 1 greedy; descending, index order within equal
//           counts) and deals it out snake-wise: position o goes to cluster
//           o mod n_cl in even rounds o / n_cl and to n_cl - 1 - (o mod n_cl)
//           in odd ones. A cluster's sequences, in round order, give its
//           row table: each sequence's target rows 0..Kb, then (sample) its
//           draft rows 0..Kb-1.
//   pass 1  As in verify_logits_kernel, over the cluster's table (each warp
//           a contiguous run of the chunks, so it changes rows rarely).
//   decide  After a cluster barrier (every CTA's ring idle) the per-row
//           partials go into every CTA's ring, a second barrier, a butterfly
//           merge; warp g decides sequence g; CTA g mod CS stores its row.
//   pass 2  The n_draw sample sequences that go on to a draw split the
//           cluster into n_draw contiguous groups of CTAs; each group runs
//           verify_logits_kernel's pass 2 over its sequence's row j with its
//           own CTAs as the cluster (totals are pushed to every CTA of the
//           cluster, so all of them agree on whether a residual fell back).
//   Every wait is bounded; no remote shared-memory access follows a CTA's
//   last cluster barrier.
#include "verify_common.cuh"

namespace sv {

constexpr int GMAX = 8;              // sequences per cluster
constexpr int GROWS = 120;           // rows per cluster
constexpr int G_MAX_CS = 16;
constexpr int KEYS = 64;             // rows read by a sequence: 0..2 * MAX_K + 1
constexpr unsigned ROW_DRAFT = 1u, ROW_SOFT = 2u;

struct GSeq {
    int b, Kb, row0, nrows;
    int sample, mode_ok, len_ok;
    // decision (identical in every CTA)
    int j, valid, use_d, bad_token;
    float u2;
    SoftPart st, sd;
};

struct GroupShared {
    uint64_t full[NSTAGE];
    uint64_t never;
    RowInfo rows[GROWS];
    float2 warp_part[NCW][GROWS];
    float2 edge_part[GROWS];
    float x_logit[GROWS];                 // the row's logit at its draft token, captured in pass 1
    float u_pos[GROWS], u2_pos[GROWS];    // Philox uniforms of the target row's position
    int row_tok_at[GROWS];                // index of the row's draft token in `tokens` (-1: none)
    unsigned char row_flags[GROWS];       // ROW_DRAFT, ROW_SOFT
    GSeq seqs[GMAX];
    float p2_part[MAX_P2_CHUNKS];
    unsigned char p2_stage[MAX_P2_CHUNKS];  // the ring stage each pass-2 chunk landed in
    float p2_edge[2];
    float2 gathered_tot[2][G_MAX_CS];     // every CTA's draw mass (float-float), by cluster rank
    int G, nrows, total_chunks, err, overflow;
    // pass 2 of this CTA's group
    ff total, tc;
    int cstar, any_retry, retry_mine;
    int found, step_lp[P2_SLOTS / 32], step_hit[P2_SLOTS / 32];
    float step_tot[P2_SLOTS / 32];
    ff tw;
};

// Two CTAs per SM: 2 x (ring + this + 1 KB reserved) within 228 KB.
static_assert(2 * (RING_BYTES + sizeof(GroupShared) + 1024) <= 228 * 1024,
              "shared state too large for two CTAs per SM");
// The ring holds the sort's scratch before pass 1 and the exchanged partials after it.
static_assert((NCW + 1) * KEYS * 4 <= RING_BYTES, "sort scratch must fit the ring");
static_assert((G_MAX_CS + 1) * GROWS * 8 <= RING_BYTES, "partials must fit the ring");

__device__ __forceinline__ float2 empty_part(bool soft) {
    return soft ? pack(SoftPart{-INFINITY, 0.0f}) : pack(ArgPart{-INFINITY, INT_MAX});
}

__device__ __forceinline__ float2 merge_part(bool soft, float2 a, float2 b) {
    return soft ? pack(merge_soft(as_soft(a), as_soft(b))) : pack(merge_arg(as_arg(a), as_arg(b)));
}

// The draft token of row r (warp-uniform r): lane l holds the tokens of rows
// l, l + 32, l + 64 and l + 96.
__device__ __forceinline__ int row_token(const int (&tok)[4], int r) {
    const int v = r < 32 ? tok[0] : r < 64 ? tok[1] : r < 96 ? tok[2] : tok[3];
    return __shfl_sync(FULL, v, r & 31);
}

// The same for a row that differs per lane (every lane takes part).
__device__ __forceinline__ int row_token_lane(const int (&tok)[4], int r) {
    const int src = r & 31;
    const int v0 = __shfl_sync(FULL, tok[0], src), v1 = __shfl_sync(FULL, tok[1], src);
    const int v2 = __shfl_sync(FULL, tok[2], src), v3 = __shfl_sync(FULL, tok[3], src);
    return r < 32 ? v0 : r < 64 ? v1 : r < 96 ? v2 : v3;
}

// Where token x lies in this CTA's pass-1 chunks of row ri (chunk -1: not in
// its interior slots here).
struct TokenSpotG {
    int chunk, byte;
};

template <typename T>
__device__ __forceinline__ TokenSpotG token_spot_g(const RowInfo& ri, int x, int c0) {
    constexpr int E = Elem<T>::E;
    TokenSpotG ts{-1, 0};
    if (x < 0) return ts;
    const int slot = (x + ri.head) / E;
    if (slot < ri.ia || slot >= ri.ib) return ts;
    ts.chunk = c0 + (slot - ri.ia) / STAGE_SLOTS;
    ts.byte = ((slot - ri.ia) % STAGE_SLOTS) * 16 + ((x + ri.head) % E) * (int)sizeof(T);
    return ts;
}

// Lane 0 writes the logit at `at` into row r's slot of every CTA of the cluster.
template <typename T>
__device__ __forceinline__ void capture_g(GroupShared& sh, cg::cluster_group& cluster, int CS, const char* at, int r) {
    float v;
    if constexpr (sizeof(T) == 4) v = *reinterpret_cast<const float*>(at);
    else v = __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(at)) << 16);
    for (int cr = 0; cr < CS; ++cr) cluster.map_shared_rank(sh.x_logit, cr)[r] = v;
}

// The chunks of the schedule one warp streams: first, first + step, ...
// below end. CHUNK_RUNS: each warp a contiguous run, so it changes rows
// rarely; else every NCW-th chunk (the CTA's warps read neighbouring chunks,
// and with a cluster's short slices a warp changes rows every chunk or two,
// each change a butterfly flush of its partial). Measured on GB300, B=64,
// K=4, V=128256 bf16 half greedy, 32 clusters of 8: 31.4 us with runs, 39.8
// with every NCW-th chunk.
constexpr bool CHUNK_RUNS = true;

struct WarpChunks {
    int first, end, step;
};

__device__ __forceinline__ WarpChunks warp_chunks(int total_chunks, int warp) {
    if (CHUNK_RUNS) {
        int ca, cb;
        split_range(total_chunks, warp, NCW, ca, cb);
        return WarpChunks{ca, cb, 1};
    }
    return WarpChunks{warp, total_chunks, NCW};
}

// The first NBUF fills of a warp's chunks.
__device__ __forceinline__ void first_fills(const VerifyParams& p, GroupShared& sh, WarpRing& wr, char* ring,
                                            const WarpChunks& wc, uint32_t seq, int lane) {
    FillCursor frc{{-1, 0, 0}, nullptr, 0, 0};
    for (int k = 0; k < NBUF; ++k) {
        const int chunk = wc.first + k * wc.step;
        if (chunk < wc.end) fill_pass1(p, sh, wr, ring, seq + k, chunk, frc, lane);
    }
}

// Pass 1 of one warp over its chunks, buffered in its NBUF stages. Writes
// one partial per row it saw.
template <typename TT, typename TD, int MS>
__device__ __forceinline__ void group_pass1(const VerifyParams& p, GroupShared& sh, WarpRing& wr, char* ring,
                                            const WarpChunks& wc, float c, int warp, int lane, uint32_t& seq,
                                            cg::cluster_group& cluster, int CS, const int (&tok)[4]) {
    constexpr bool CAN_SAMPLE = (MS & MS_SAMPLE) != 0, CAN_GREEDY = (MS & MS_GREEDY) != 0;
    constexpr bool SAME = std::is_same<TT, TD>::value;
    RowCursor rc{-1, 0, 0};
    FillCursor frc{{-1, 0, 0}, nullptr, 0, 0};  // the refills' chunks only increase
    int cur_row = -1, ia = 0, ib = 0, head = 0;
    bool soft = !CAN_GREEDY, draft = false;
    TokenSpotG ts{-1, 0};
    SoftAcc sa = soft_acc_empty();
    ArgAcc aa = arg_acc_empty();
    auto flush = [&]() {
        if (cur_row < 0) return;
        if (CAN_SAMPLE && soft) {
            flush_row<TT, true>(sh, warp, lane, cur_row, sa, aa, head);
        } else if constexpr (CAN_GREEDY) {
            // greedy rows are target rows
            flush_row<TT, false>(sh, warp, lane, cur_row, sa, aa, head);
        }
    };
    for (int chunk = wc.first; chunk < wc.end; chunk += wc.step, ++seq) {
        seek_row(rc, sh.rows, chunk);
        if (rc.r != cur_row) {  // a new row: flush the last one, look the new one up once
            flush();
            sa = soft_acc_empty();
            aa = arg_acc_empty();
            cur_row = rc.r;
            const RowInfo ri = sh.rows[cur_row];
            ia = ri.ia;
            ib = ri.ib;
            head = ri.head;
            const unsigned fl = sh.row_flags[cur_row];
            draft = (fl & ROW_DRAFT) != 0;
            soft = CAN_SAMPLE && (!CAN_GREEDY || (fl & ROW_SOFT) != 0);
            ts = TokenSpotG{-1, 0};
            const int x = row_token(tok, cur_row);
            if (soft) ts = (SAME || !draft) ? token_spot_g<TT>(ri, x, rc.c0) : token_spot_g<TD>(ri, x, rc.c0);
        }
        if (!wr.wait(sh, seq)) {
            atomicExch(&sh.err, 1);
            break;
        }
        const int q0 = ia + (chunk - rc.c0) * STAGE_SLOTS;
        const int n = min(STAGE_SLOTS, ib - q0);
        const char* stage = wr.stage(ring, seq);
        uint4 d[CHUNK_LANE_SLOTS];
        if (n == STAGE_SLOTS) {  // a full chunk (warp-uniform): no per-slot select
#pragma unroll
            for (int u = 0; u < CHUNK_LANE_SLOTS; ++u) d[u] = lds128(stage + (u * 32 + lane) * 16);
        } else {  // slots past the chunk's end read as -inf of the row's own type
            const uint4 pad = (SAME || !draft) ? neg_inf_slot<TT>() : neg_inf_slot<TD>();
#pragma unroll
            for (int u = 0; u < CHUNK_LANE_SLOTS; ++u) {
                const int i = u * 32 + lane;
                d[u] = i < n ? lds128(stage + i * 16) : pad;
            }
        }
        if (chunk == ts.chunk && lane == 0) {
            if (SAME || !draft) capture_g<TT>(sh, cluster, CS, stage + ts.byte, cur_row);
            else capture_g<TD>(sh, cluster, CS, stage + ts.byte, cur_row);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (chunk + NBUF * wc.step < wc.end)
            fill_pass1(p, sh, wr, ring, seq + NBUF, chunk + NBUF * wc.step, frc, lane);
        if (CAN_SAMPLE && soft) {
            if (SAME || !draft) reduce_chunk<TT, true>(sa, aa, d, n, q0, c, lane);
            else reduce_chunk<TD, true>(sa, aa, d, n, q0, c, lane);
        } else if constexpr (CAN_GREEDY) {
            reduce_chunk<TT, false>(sa, aa, d, n, q0, c, lane);
        }
    }
    flush();
}

// The partial slots at the two ends of this CTA's slice of row r (lane 0 the
// low end, lane 1 the high end), reduced like the chunks; captures the draft
// token's logit when it lies in one of them.
template <typename T, bool SOFT>
__device__ __forceinline__ float2 group_edge(const VerifyParams& p, GroupShared& sh, const RowInfo& ri, int r, int x,
                                             int V, float c, int lane, cg::cluster_group& cluster, int CS) {
    constexpr int E = Elem<T>::E;
    const RowGeom g{ri.base, ri.head, 0};
    const T* row = reinterpret_cast<const T*>(ri.base) + ri.head;
    uint4 d[1];
    int qs[1];
    qs[0] = lane == 0 ? ri.edge_lo : lane == 1 ? ri.edge_hi : -1;
    d[0] = qs[0] >= 0 ? load_slot<T>(p, g, row, V, qs[0]) : neg_inf_slot<T>();
    if (SOFT) {
        if (x >= 0 && qs[0] >= 0 && (x + ri.head) / E == qs[0]) {
            const float v = elem_rt<T>(d[0], (x + ri.head) % E);
            for (int cr = 0; cr < CS; ++cr) cluster.map_shared_rank(sh.x_logit, cr)[r] = v;
        }
        SoftAcc ea = soft_acc_empty();
        soft_group<T, 1>(ea, d, c);
        SoftPart pp{ea.R, soft_acc_sum(ea)};
        if (ea.R == -INFINITY) pp.s = 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            pp = merge_soft(pp, SoftPart{__shfl_xor_sync(FULL, pp.R, o), __shfl_xor_sync(FULL, pp.s, o)});
        return pack(pp);
    } else {
        ArgPart ea{-INFINITY, INT_MAX};
        arg_group<T, 1>(ea, d, qs, ri.head);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ea = merge_arg(ea, ArgPart{__shfl_xor_sync(FULL, ea.v, o), __shfl_xor_sync(FULL, ea.i, o)});
        return pack(ea);
    }
}

// The cluster total of one pass-2 group (CTAs lo .. lo + n - 1) and the CTA
// whose mass holds t = u2 * total: an inclusive float-float scan over lanes
// cr < n, as verify_logits_kernel does over its cluster. Called by a whole warp.
__device__ __forceinline__ void group_draw_scan(const GroupShared& sh, int attempt, int lo, int n, float u2, int lane,
                                                ff& S, int& cstar, ff& tc) {
    const float2 g = lane < n ? sh.gathered_tot[attempt][lo + lane] : make_float2(0.0f, 0.0f);
    const ff v{g.x, g.y};
    ff incl = v;
#pragma unroll
    for (int o = 1; o < MAX_CS; o <<= 1) {
        const ff y = ff_shfl_up(incl, o);
        if (lane >= o) incl = ff_add(y, incl);
    }
    S = ff_shfl(incl, MAX_CS - 1);
    const ff t = ff_mul(S, u2);
    const unsigned hit = __ballot_sync(FULL, lane < n && ff_gt(incl, t));
    const unsigned pos = __ballot_sync(FULL, lane < n && v.hi > 0.0f);
    const ff excl = ff_add(incl, ff_neg(v));
    if (hit) {
        cstar = __ffs(hit) - 1;
        tc = ff_shfl(ff_add(t, ff_neg(excl)), cstar);
    } else {  // t at or past the summed mass: take the last positive element
        cstar = pos ? 31 - __clz(pos) : -1;
        tc = ff{INFINITY, 0.0f};
    }
}

template <typename TT, typename TD, int MS>
__global__ void __launch_bounds__(NTHREADS, 2) verify_grouped_kernel(VerifyParams p) {
    constexpr bool CAN_SAMPLE = (MS & MS_SAMPLE) != 0, CAN_GREEDY = (MS & MS_GREEDY) != 0;
    constexpr bool SAME = std::is_same<TT, TD>::value;
    extern __shared__ __align__(128) char ring[];
    __shared__ GroupShared sh;
    launch_dependents();
    cluster_arrive_started();
    cg::cluster_group cluster = cg::this_cluster();
    const int CS = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_cl = (int)(gridDim.x / CS), cl = (int)(blockIdx.x / CS);
    const int B = p.B, K = p.K, V = p.V;
    const float c = p.c;
    const TT* tgt = static_cast<const TT*>(p.target);
    const TD* drf = static_cast<const TD*>(p.draft);
    // A plain call: no input is read before the work ahead of it on the
    // stream has completed (the wait returns at once unless the launch allows
    // an early start).
    const bool prologue_reads = p.modes != nullptr || p.draft_lens != nullptr;
    if (prologue_reads) grid_dependency_wait();

    // ---------------- assign: this cluster's sequences ----------------
    // thread t looks at sequence t (B <= NTHREADS)
    int Kb_t = K, rows_t = 0;
    bool sample_t = false, mode_ok_t = false, len_ok_t = false;
    if (tid < B) {
        const int mode = p.modes ? ld_in(p, p.modes + tid, -1) : p.mode;
        Kb_t = p.draft_lens ? ld_in(p, p.draft_lens + tid, -1) : K;
        len_ok_t = Kb_t >= 0 && Kb_t <= K;
        mode_ok_t = (mode == 0 || mode == 1) && !(mode == 1 && drf == nullptr) && len_ok_t;
        sample_t = CAN_SAMPLE && (!CAN_GREEDY || mode == 1) && mode_ok_t;
        rows_t = mode_ok_t ? (sample_t ? 2 * Kb_t + 1 : Kb_t + 1) : 0;
    }
    int pos = tid;  // every sequence reads the same rows: index order
    if (prologue_reads) {
        // stable counting sort by rows, descending (keys 63 - rows)
        int* wh = reinterpret_cast<int*>(ring);  // [NCW][KEYS] counts per warp
        int* kbase = wh + NCW * KEYS;            // [KEYS] first position of each key
        for (int i = tid; i < NCW * KEYS; i += NTHREADS) wh[i] = 0;
        __syncthreads();
        const int key = tid < B ? KEYS - 1 - rows_t : KEYS;
        const unsigned same = __match_any_sync(FULL, key);
        const int below = __popc(same & ((1u << lane) - 1u));
        if (tid < B && below == 0) wh[warp * KEYS + key] = __popc(same);
        __syncthreads();
        if (warp == 0) {
            int t0 = 0, t1 = 0;
            for (int w = 0; w < NCW; ++w) {
                t0 += wh[w * KEYS + lane];
                t1 += wh[w * KEYS + 32 + lane];
            }
            int i0 = t0, i1 = t1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y0 = __shfl_up_sync(FULL, i0, o), y1 = __shfl_up_sync(FULL, i1, o);
                if (lane >= o) {
                    i0 += y0;
                    i1 += y1;
                }
            }
            const int T0 = __shfl_sync(FULL, i0, 31);
            kbase[lane] = i0 - t0;
            kbase[32 + lane] = T0 + i1 - t1;
        }
        __syncthreads();
        if (tid < B) {
            int before = 0;
            for (int w = 0; w < warp; ++w) before += wh[w * KEYS + key];
            pos = kbase[key] + before + below;
        }
        // the ring is next written by bulk copies
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        int G = 0;
        for (int g = 0;; ++g) {
            const int o = g * n_cl + ((g & 1) ? n_cl - 1 - cl : cl);
            if (o >= B) break;
            ++G;
        }
        sh.overflow = G > GMAX;
        sh.G = min(G, GMAX);
        sh.err = 0;
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&sh.full[s], 1);
        mbar_init(&sh.never, 1);
        fence_barrier_init();
    }
    if (tid < B) {
        const int g = pos / n_cl, col = pos % n_cl;
        if (((g & 1) ? n_cl - 1 - col : col) == cl && g < GMAX) {
            GSeq& s = sh.seqs[g];
            s.b = tid;
            s.Kb = Kb_t;
            s.nrows = rows_t;
            s.sample = sample_t;
            s.mode_ok = mode_ok_t;
            s.len_ok = len_ok_t;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int r0 = 0;
        for (int g = 0; g < sh.G; ++g) {
            GSeq& s = sh.seqs[g];
            if (r0 + s.nrows > GROWS) {  // (the host's plan never gets here)
                s.nrows = 0;
                s.mode_ok = 0;
                sh.overflow = 1;
            }
            s.row0 = r0;
            r0 += s.nrows;
        }
        sh.nrows = r0;
    }
    __syncthreads();
    const int G = sh.G, nrows = sh.nrows;
    // the row table: sequence g's target rows 0..Kb, then its draft rows
    if (tid < nrows) {
        int g = 0;
        while (g + 1 < G && tid >= sh.seqs[g + 1].row0) ++g;
        const GSeq s = sh.seqs[g];
        const int i = tid - s.row0;
        const bool draft = i > s.Kb;
        sh.rows[tid] = draft ? make_row_info<TD>(draft_row(drf, s.b, K, V, i - s.Kb - 1), V, rank, CS)
                             : make_row_info<TT>(target_row(tgt, s.b, K, V, i), V, rank, CS);
        sh.row_flags[tid] = (unsigned char)((draft ? ROW_DRAFT : 0u) | (s.sample ? ROW_SOFT : 0u));
        sh.row_tok_at[tid] = draft ? s.b * K + (i - s.Kb - 1) : (i < s.Kb ? s.b * K + i : -1);
        const bool soft = CAN_SAMPLE && (!CAN_GREEDY || s.sample);
        sh.edge_part[tid] = empty_part(soft);
        for (int w = 0; w < NCW; ++w) sh.warp_part[w][tid] = empty_part(soft);
    }
    __syncthreads();
    if (warp == 0) {
        // prefix sums of the rows' chunk counts (the pass-1 schedule)
        int cnt = 0;
        for (int r0 = 0; r0 < nrows; r0 += 32) {
            const int r = r0 + lane;
            const int m = r < nrows ? (sh.rows[r].ib - sh.rows[r].ia + STAGE_SLOTS - 1) / STAGE_SLOTS : 0;
            int incl = m;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += y;
            }
            if (r < nrows) sh.rows[r].c1 = cnt + incl;
            cnt += __shfl_sync(FULL, incl, 31);
        }
        if (lane == 0) sh.total_chunks = cnt;
    }
    __syncthreads();
    const int total_chunks = sh.total_chunks;

    // ---------------- pass 1 ----------------
    if (!prologue_reads) grid_dependency_wait();  // the first input read follows
    WarpRing wr{warp, 0u, 0u};
    uint32_t seq = 0;
    const WarpChunks wc = warp_chunks(total_chunks, warp);
    first_fills(p, sh, wr, ring, wc, seq, lane);
    // while the first copies are in flight: the draft tokens of the rows
    // (lane l: rows l, l + 32, ...) and, in warp g, sequence g's uniforms
    int tok[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = k * 32 + lane;
        const int at = r < nrows ? sh.row_tok_at[r] : -1;
        tok[k] = at >= 0 ? ld_in(p, p.tokens + at, -1) : -1;
    }
    if (CAN_SAMPLE && warp < G) {
        const GSeq s = sh.seqs[warp];
        if (s.sample && lane <= s.Kb) {
            const uint64_t seqid = p.seq_ids ? ld_in(p, p.seq_ids + s.b, (uint64_t)s.b) : (uint64_t)s.b;
            position_uniforms(p.seed, seqid, (uint32_t)lane, sh.u_pos[s.row0 + lane], sh.u2_pos[s.row0 + lane]);
        }
    }
    cluster_wait_started();  // pass 1 writes the captured logits into every CTA of the cluster
    group_pass1<TT, TD, MS>(p, sh, wr, ring, wc, c, warp, lane, seq, cluster, CS, tok);
    // the partial slots at the slices' ends (rows not 16-byte aligned)
    for (int r = warp; r < nrows; r += NCW) {
        const RowInfo ri = sh.rows[r];
        if (ri.edge_lo < 0 && ri.edge_hi < 0) continue;
        const unsigned fl = sh.row_flags[r];
        const bool draft = (fl & ROW_DRAFT) != 0;
        const bool soft = CAN_SAMPLE && (!CAN_GREEDY || (fl & ROW_SOFT) != 0);
        const int x = soft ? row_token(tok, r) : -1;
        float2 part;
        if (CAN_SAMPLE && soft) {
            part = (SAME || !draft) ? group_edge<TT, true>(p, sh, ri, r, x, V, c, lane, cluster, CS)
                                    : group_edge<TD, true>(p, sh, ri, r, x, V, c, lane, cluster, CS);
        } else {
            part = group_edge<TT, false>(p, sh, ri, r, x, V, c, lane, cluster, CS);
        }
        if (lane == 0) sh.edge_part[r] = part;
    }
    if (p.test_wait_timeout && tid == 0 && !mbar_wait(&sh.never, 0, 1u << 12)) atomicExch(&sh.err, 1);
    wr.drain(sh);  // no copy of this CTA is in flight past this point
    __syncthreads();
    cluster.sync();  // every CTA's ring is idle: the partials may go there

    // ---------------- exchange, merge ----------------
    float2* gathered = reinterpret_cast<float2*>(ring);  // [G_MAX_CS][GROWS]
    float2* merged = gathered + G_MAX_CS * GROWS;        // [GROWS]
    const bool poison = sh.err != 0;
    for (int t = tid; t < CS * nrows; t += NTHREADS) {
        const int dst = t / nrows, r = t % nrows;
        const bool soft = CAN_SAMPLE && (!CAN_GREEDY || (sh.row_flags[r] & ROW_SOFT) != 0);
        float2 acc = sh.edge_part[r];
        for (int w = 0; w < NCW; ++w) acc = merge_part(soft, acc, sh.warp_part[w][r]);
        if (poison) acc = make_float2(__int_as_float(0x7fc00000), 0.0f);  // poison: invalid
        cluster.map_shared_rank(gathered, dst)[rank * GROWS + r] = acc;
    }
    cluster.sync();
    {
        const int rows_per_pass = 32 / CS;
        const int r_in = lane / CS, cr = lane % CS;
        for (int r0 = warp * rows_per_pass; r0 < nrows; r0 += NCW * rows_per_pass) {
            const int r = r0 + r_in;
            // the rows of one pass may differ in kind; each lane group merges its own
            const bool soft = r < nrows && CAN_SAMPLE && (!CAN_GREEDY || (sh.row_flags[r] & ROW_SOFT) != 0);
            float2 acc = r < nrows ? gathered[cr * GROWS + r] : empty_part(soft);
            for (int o = CS >> 1; o > 0; o >>= 1) {
                const float2 other = make_float2(__shfl_xor_sync(FULL, acc.x, o), __shfl_xor_sync(FULL, acc.y, o));
                acc = merge_part(soft, acc, other);
            }
            if (cr == 0 && r < nrows) merged[r] = acc;
        }
    }
    __syncthreads();

    // ---------------- decide: warp g, sequence g (in every CTA) ----------------
    if (warp < G) {
        GSeq& s = sh.seqs[warp];
        const int b = s.b, Kb = s.Kb, row0 = s.row0;
        const bool mode_ok = s.mode_ok != 0, sample = s.sample != 0;
        const bool use_soft = !CAN_GREEDY || (CAN_SAMPLE && sample);
        const int nr = mode_ok ? s.nrows : 0;
        bool bad = !mode_ok;
        for (int r = lane; r < nr; r += 32) {
            const float2 acc = merged[row0 + r];
            if (use_soft) {
                const SoftPart sp = as_soft(acc);
                bad |= !(isfinite(sp.R) && isfinite(sp.s) && sp.s > 0.0f);
            } else {
                const ArgPart ap = as_arg(acc);
                bad |= !isfinite(ap.v) || ap.i < 0 || ap.i >= V;
            }
        }
        const int x_all = row_token_lane(tok, row0 + min(lane, 31));
        float u = 0.0f, u2 = 0.0f;
        if (sample && lane <= Kb) {
            u = sh.u_pos[row0 + lane];
            u2 = sh.u2_pos[row0 + lane];
        }
        int x = -1;
        bool bad_token = false, rej = false;
        float et = 0.0f, ed = 0.0f, St = 1.0f, Sd = 1.0f;
        if (mode_ok && lane < Kb) {
            x = x_all;
            bad_token = x < 0 || x >= V;
            if (!bad_token) {
                if (!use_soft) {
                    rej = x != as_arg(merged[row0 + lane]).i;
                } else {
                    const SoftPart st = as_soft(merged[row0 + lane]);
                    const SoftPart sd = as_soft(merged[row0 + Kb + 1 + lane]);
                    et = ex2(fmaf(sh.x_logit[row0 + lane], c, -st.R));
                    ed = ex2(fmaf(sh.x_logit[row0 + Kb + 1 + lane], c, -sd.R));
                    St = st.s;
                    Sd = sd.s;
                    rej = !accept_draft(u, ed, St, et, Sd);
                }
            }
        }
        const bool any_bad_token = __any_sync(FULL, bad_token);
        const bool invalid = __any_sync(FULL, bad) || any_bad_token;
        const unsigned rejm = __ballot_sync(FULL, rej);
        const int j = rejm ? __ffs(rejm) - 1 : (mode_ok ? Kb : 0);
        const float u2j = __shfl_sync(FULL, u2, j & 31);
        if (lane == 0) {
            s.j = j;
            s.valid = !invalid;
            s.bad_token = any_bad_token;
            s.u2 = u2j;
            s.use_d = 0;
            if (sample && !invalid) {
                s.st = as_soft(merged[row0 + j]);
                s.use_d = j < Kb;
                s.sd = j < Kb ? as_soft(merged[row0 + Kb + 1 + j]) : SoftPart{-INFINITY, 0.0f};
            }
        }
        if (rank == warp % CS) {  // this CTA stores sequence g's row
            const int greedy_tok = (!sample && !invalid) ? as_arg(merged[row0 + j]).i : -1;
            if (lane <= K) {
                int tk = -1;
                if (!invalid) tk = lane < j ? x : (lane == j ? greedy_tok : -1);
                // in sample mode position j belongs to the CTA that finds the draw
                if (!(sample && !invalid && lane == j)) st_out(p, p.out_tokens + ((size_t)b * (K + 1) + lane), tk);
            }
            if (lane == 0) st_out(p, p.out_n_accepted + (b), invalid ? -1 : j);
            if (lane < K) {
                const float qnan = __int_as_float(0x7fc00000);
                const bool tested = sample && !invalid && lane < Kb;
                if (p.out_p_target) st_out(p, p.out_p_target + ((size_t)b * K + lane), tested ? et / St : qnan);
                if (p.out_p_draft) st_out(p, p.out_p_draft + ((size_t)b * K + lane), tested ? ed / Sd : qnan);
            }
            if (lane == 0 && (!sample || invalid) && p.out_residual_mass)
                st_out(p, p.out_residual_mass + (b), __int_as_float(0x7fc00000));
            if (lane < 2 && (!sample || invalid) && p.out_draw_edges)
                st_out(p, p.out_draw_edges + (2 * (size_t)b + lane), __int_as_float(0x7fc00000));
            if (lane == 0 && p.status_word && invalid)
                atomicOr(p.status_word, !s.len_ok      ? (unsigned)SV_FLAG_BAD_LENGTH
                                        : !mode_ok     ? (unsigned)SV_FLAG_BAD_MODE
                                        : any_bad_token ? (unsigned)SV_FLAG_BAD_TOKEN
                                                        : (unsigned)SV_FLAG_BAD_ROW);
            if (lane == 0 && p.status_word && sh.err) atomicOr(p.status_word, (unsigned)SV_FLAG_TIMEOUT);
        }
    }
    if (tid == 0 && rank == 0 && sh.overflow && p.status_word) atomicOr(p.status_word, (unsigned)SV_FLAG_BAD_ROW);
    __syncthreads();

    // ---------------- pass 2: one group of CTAs per drawing sequence ----------------
    int n_draw = 0, my_s = -1, lo = 0, hi = 0;
    if (CAN_SAMPLE) {
        for (int g = 0; g < G; ++g) n_draw += sh.seqs[g].sample && sh.seqs[g].valid;
        for (int s = 0; s < n_draw; ++s) {
            int a, e;
            split_range(CS, s, n_draw, a, e);
            if (rank >= a && rank < e) {
                my_s = s;
                lo = a;
                hi = e;
            }
        }
    }
    if (!CAN_SAMPLE || n_draw == 0) {
        wr.drain(sh);
        return;  // every remote access of this CTA's shared memory happened before the last barrier
    }
    // (n_draw <= G <= CS, so every group has a CTA and my_s >= 0)
    int gs = -1;
    for (int g = 0, s = 0; g < G; ++g) {
        if (sh.seqs[g].sample && sh.seqs[g].valid) {
            if (s == my_s) gs = g;
            ++s;
        }
    }
    const GSeq me = sh.seqs[gs];
    const int b = me.b, j = me.j;
    const int sub_rank = rank - lo, sub_cs = hi - lo;
    DrawSrc<TT, TD> src;
    src.trow = tgt + ((size_t)b * (K + 1) + j) * V;
    src.drow = me.use_d ? drf + ((size_t)b * K + j) * V : reinterpret_cast<const TD*>(src.trow);
    src.gt = row_geom(src.trow, V);
    src.gd = row_geom(src.drow, V);
    src.V = V;
    src.same_slots = SAME && src.gd.head == src.gt.head;
    int qa, qb;
    split_range(src.gt.nslot, sub_rank, sub_cs, qa, qb);
    const WarpSlots sl = warp_slots<TT>(src.gt, V, qa, qb);
    const bool draft_in_ring = src.same_slots;
    constexpr bool SPAN_TYPES = sizeof(TT) == 4 && sizeof(TD) == 2;
    const uint32_t span_off = SPAN_TYPES ? draft_span<TT, TD>(src, sl.ia, 0).off : 0u;
    DrawRows w;
    w.c = c;
    w.ntR = -me.st.R;
    w.invSt = 1.0f / me.st.s;
    w.ndR = -me.sd.R;
    w.invSd = me.use_d ? 1.0f / me.sd.s : 0.0f;
    pack_draw_rows(w);
    const int n_chunks = (sl.ib - sl.ia + P2_SLOTS - 1) / P2_SLOTS;
    constexpr int STEPS = P2_SLOTS / 32;
    fence_proxy_async_smem();  // the ring, last written through generic stores, takes bulk copies again
    __syncthreads();
    bool fell_back = false;  // this group's residual summed to zero: it draws again from P_t
    for (int attempt = 0;; ++attempt) {
        // a group that does not go again keeps its first attempt (its parts,
        // its stages and its draw rows) for the search
        const bool active = attempt == 0 || fell_back;
        if (active) w.use_d = me.use_d && attempt == 0;
        const bool ring_d = w.use_d && draft_in_ring;
        const bool span_d = SPAN_TYPES && w.use_d;
        if (active && !sh.err) {
            for (int jj = 0; jj < NBUF; ++jj) {
                const int ci = warp + NCW * jj;
                if (ci < n_chunks) fill_pass2<TT, TD>(p, sh, wr, ring, seq + jj, src, sl.ia, sl.ib, ci, ring_d, span_d, lane);
            }
            for (int ci = warp; ci < n_chunks; ci += NCW) {
                const int q = sl.ia + ci * P2_SLOTS;
                const int n = min(P2_SLOTS, sl.ib - q);
                uint4 dt[STEPS], dd[STEPS];
                if (!wr.wait(sh, seq)) {
                    atomicExch(&sh.err, 1);
                    break;
                }
                const char* stage = wr.stage(ring, seq);
                if (lane == 0) sh.p2_stage[ci] = (unsigned char)(warp + NCW * (int)(seq % NBUF));
#pragma unroll
                for (int kk = 0; kk < STEPS; ++kk) {
                    const int i = kk * 32 + lane;
                    dt[kk] = neg_inf_slot<TT>();
                    dd[kk] = neg_inf_slot<TT>();
                    if (i < n) {
                        dt[kk] = lds128(stage + i * 16);
                        if (ring_d) dd[kk] = lds128(stage + P2_DRAFT_OFF + i * 16);
                        if (span_d) dd[kk] = span_slot(stage + P2_DRAFT_OFF, span_off, i);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (ci + NBUF * NCW < n_chunks)
                    fill_pass2<TT, TD>(p, sh, wr, ring, seq + NBUF, src, sl.ia, sl.ib, ci + NBUF * NCW, ring_d, span_d,
                                       lane);
                ++seq;
                // the chunk's draw mass: per lane over its slots, then one warp sum
                f32x2 acc = 0ull;
#pragma unroll
                for (int kk = 0; kk < STEPS; ++kk) {
                    const int i = kk * 32 + lane;
                    if (w.use_d && !draft_in_ring && !span_d && i < n)
                        dd[kk] = load_elems_as<TT, TD>(p, src.drow, V, (q + i) * Elem<TT>::E - src.gt.head);
#pragma unroll
                    for (int k2 = 0; k2 < Elem<TT>::E / 2; ++k2)
                        acc = add2(acc, draw_mass2(w, slot_pair<TT>(dt[kk], k2), slot_pair<TT>(dd[kk], k2)));
                }
                float a0, a1;
                unpack2(acc, a0, a1);
                float part = a0 + a1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
                if (lane == 0) sh.p2_part[ci] = part;
            }
            if (warp == 0) {
                // the partial slots at the two ends of this CTA's slice
                float e_lo = 0.0f, e_hi = 0.0f;
                if (sl.edge_lo >= 0 || sl.edge_hi >= 0) {
                    uint4 dt, dd;
                    const int q = lane == 0 ? sl.edge_lo : lane == 1 ? sl.edge_hi : -1;
                    load_draw_slot<TT, TD>(p, src, w.use_d, q, dt, dd);
                    const float m = slot_mass<TT>(w, dt, dd);
                    e_lo = __shfl_sync(FULL, m, 0);
                    e_hi = __shfl_sync(FULL, m, 1);
                }
                if (lane == 0) {
                    sh.p2_edge[0] = e_lo;
                    sh.p2_edge[1] = e_hi;
                }
            }
        }
        __syncthreads();
        // this CTA's draw mass (float-float), pushed to every CTA of the cluster
        if (warp == 0) {
            ff t = ff_from(0.0f);
            for (int i = lane; i < n_chunks; i += 32) t = ff_add(t, sh.p2_part[i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t = ff_add(t, ff_shfl_xor(t, o));
            t = ff_add(ff_add(t, sh.p2_edge[0]), sh.p2_edge[1]);
            if (sh.err) t = ff_from(0.0f);
            t = ff_shfl(t, 0);  // one value for every destination CTA
            if (lane < CS) cluster.map_shared_rank(&sh.gathered_tot[0][0], lane)[attempt * G_MAX_CS + rank] = make_float2(t.hi, t.lo);
        }
        cluster.sync();
        // Every CTA scans every group (identical inputs, identical code), so
        // all agree on which groups' residuals summed to zero and go again
        // with P_t of row j.
        if (warp == 0) {
            int retry_any = 0, retry_me = 0;
            const bool retried_before = attempt > 0 && sh.retry_mine;  // read before lane 0 rewrites it
            for (int g = 0, s = 0; g < G; ++g) {
                const GSeq& o = sh.seqs[g];
                if (!(o.sample && o.valid)) continue;
                int a, e;
                split_range(CS, s, n_draw, a, e);
                ff S, tc;
                int cstar;
                group_draw_scan(sh, attempt, a, e - a, o.u2, lane, S, cstar, tc);
                const bool was_active = attempt == 0 || (s == my_s && retried_before);
                const bool retry = attempt == 0 && o.use_d && !(S.hi > 0.0f);
                retry_any |= retry;
                if (s == my_s) {
                    retry_me = retry;
                    if (was_active && lane == 0) {
                        sh.total = S;
                        sh.cstar = cstar;
                        sh.tc = tc;
                    }
                }
                ++s;
            }
            if (lane == 0) {
                sh.any_retry = retry_any;
                sh.retry_mine = retry_me;
            }
        }
        __syncthreads();
        if (!sh.any_retry) break;
        // Some group's residual summed to zero in float: that group falls
        // back to P_t of row j (reported at the end); the others keep theirs.
        fell_back = sh.retry_mine != 0;
    }

    if (sub_rank == sh.cstar) {  // the CTA holding the draw (uniform over the CTA)
        if (warp == 0) {
            // Walk down this CTA's parts in index order (low edge slot, the
            // chunk parts, high edge slot): each lane sums a contiguous run of
            // parts, a warp scan finds the run holding tc, its lane walks it.
            const int P = n_chunks + 2;
            auto part_val = [&](int i) -> float {
                if (i == 0) return sh.p2_edge[0];
                if (i == P - 1) return sh.p2_edge[1];
                return sh.p2_part[i - 1];
            };
            const int per = (P + 31) / 32;
            const int i0 = min(P, lane * per), i1 = min(P, i0 + per);
            ff mine = ff_from(0.0f);
            int last_pos = -1;
            for (int i = i0; i < i1; ++i) {
                const float v = part_val(i);
                mine = ff_add(mine, v);
                if (v > 0.0f) last_pos = i;
            }
            ff incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const ff y = ff_shfl_up(incl, o);
                if (lane >= o) incl = ff_add(y, incl);
            }
            const ff tc = sh.tc;
            const bool tc_inf = isinf(tc.hi);
            const unsigned hit = __ballot_sync(FULL, !tc_inf && ff_gt(incl, tc));
            int found = -1;
            ff tw{INFINITY, 0.0f};
            if (hit) {
                const int l = __ffs(hit) - 1;
                if (lane == l) {
                    ff t = ff_add(tc, ff_neg(ff_add(incl, ff_neg(mine))));
                    for (int i = i0; i < i1; ++i) {
                        const float v = part_val(i);
                        if (ff_gt(ff_from(v), t)) { found = i; tw = t; break; }
                        t = ff_add(t, -v);
                    }
                    if (found < 0) found = last_pos;  // rounding: this run's last positive part
                }
                found = __shfl_sync(FULL, found, l);
                tw = ff_shfl(tw, l);
            }
            if (found < 0) {  // rounding put tc past every part: the last positive part
                int lp = last_pos;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(FULL, lp, o));
                found = lp;
                tw = ff{INFINITY, 0.0f};
            }
            if (lane == 0) {
                sh.found = found;
                sh.tw = tw;
            }
        }
        __syncthreads();
        // Inverse CDF inside the part: warp k takes its k-th step of 32 slots
        // (all loaded at once); the first step whose running mass passes tw
        // holds the token.
        const int found = sh.found;
        if (found >= 0) {
            const int P = n_chunks + 2;
            int q0, n;
            if (found == 0) { q0 = sl.edge_lo; n = 1; }
            else if (found == P - 1) { q0 = sl.edge_hi; n = 1; }
            else {
                q0 = sl.ia + (found - 1) * P2_SLOTS;
                n = min(P2_SLOTS, sl.ib - q0);
            }
            const ff tw = sh.tw;
            const bool tw_inf = isinf(tw.hi);
            // When no stage was refilled during pass 2 (at most NSTAGE
            // chunks), the part's chunk is still in its stage: the search
            // takes it from there instead of reading the row again.
            const bool in_ring = n_chunks <= NSTAGE && found > 0 && found < P - 1 && !sh.err;
            DrawStep<TT, TD> st;
            if (warp < STEPS) {
                if (in_ring) {
                    const char* stage = ring + (size_t)sh.p2_stage[found - 1] * STAGE_BYTES;
                    const int i = warp * 32 + lane;
                    const int q = i < n ? q0 + i : -1;
                    uint4 dt = neg_inf_slot<TT>(), dd = neg_inf_slot<TT>();
                    if (i < n) {
                        dt = lds128(stage + i * 16);
                        if (w.use_d && draft_in_ring) dd = lds128(stage + P2_DRAFT_OFF + i * 16);
                        else if (SPAN_TYPES && w.use_d) dd = span_slot(stage + P2_DRAFT_OFF, span_off, i);
                        else if (w.use_d) dd = load_elems_as<TT, TD>(p, src.drow, V, q * Elem<TT>::E - src.gt.head);
                    }
                    st.take(w, dt, dd, q, src.gt.head, lane);
                } else {
                    st.load(p, src, w, q0, n, warp, lane);
                }
                if (lane == 0) {
                    sh.step_tot[warp] = st.tot;
                    sh.step_lp[warp] = st.last_pos;
                }
            }
            __syncthreads();
            ff run = ff_from(0.0f);
            if (warp < STEPS) {
                for (int k = 0; k < warp; ++k) run = ff_add(run, sh.step_tot[k]);
                const unsigned hit = __ballot_sync(FULL, !tw_inf && ff_gt(ff_add(run, st.incl), tw));
                if (lane == 0) sh.step_hit[warp] = hit ? __ffs(hit) - 1 : -1;
            }
            __syncthreads();
            int kstar = -1;
            for (int k = STEPS - 1; k >= 0; --k)
                if (sh.step_hit[k] >= 0) kstar = k;
            if (kstar >= 0 && warp == kstar) {
                const int l = sh.step_hit[kstar];
                float d0, d1;
                const int token = st.walk(run, tw, l, d0, d1);
                if (lane == l) {
                    st_out(p, p.out_tokens + ((size_t)b * (K + 1) + j), token);
                    if (p.out_draw_edges) {
                        st_out(p, p.out_draw_edges + (2 * (size_t)b), d0);
                        st_out(p, p.out_draw_edges + (2 * (size_t)b + 1), d1);
                    }
                }
            } else if (kstar < 0 && tid == 0) {
                int lp = -1;  // tw past the part's mass: its last positive element
                for (int k = 0; k < STEPS; ++k) lp = max(lp, sh.step_lp[k]);
                st_out(p, p.out_tokens + ((size_t)b * (K + 1) + j), lp);
                if (p.out_draw_edges) {
                    st_out(p, p.out_draw_edges + (2 * (size_t)b), 0.0f);
                    st_out(p, p.out_draw_edges + (2 * (size_t)b + 1), 0.0f);
                }
            }
        }
    }

    // The group's first CTA: its sequence's flags and residual mass.
    if (sub_rank == 0 && tid == 0) {
        if (p.status_word && fell_back) atomicOr(p.status_word, (unsigned)SV_FLAG_RESIDUAL_FALLBACK);
        if (sh.cstar >= 0 && isinf(sh.tc.hi) && p.status_word) atomicOr(p.status_word, (unsigned)SV_FLAG_DRAW_EDGE);
        if (sh.cstar < 0) {
            // No mass at all (cannot happen for a valid row): report the
            // sequence as invalid rather than leave a slot unwritten.
            st_out(p, p.out_tokens + ((size_t)b * (K + 1) + j), -1);
            st_out(p, p.out_n_accepted + (b), -1);
            if (p.out_draw_edges) {
                st_out(p, p.out_draw_edges + (2 * (size_t)b), __int_as_float(0x7fc00000));
                st_out(p, p.out_draw_edges + (2 * (size_t)b + 1), __int_as_float(0x7fc00000));
            }
            if (p.status_word) atomicOr(p.status_word, (unsigned)SV_FLAG_BAD_ROW);
        }
        if (p.out_residual_mass) st_out(p, p.out_residual_mass + (b), sh.total.hi + sh.total.lo);
        if (p.status_word && sh.err) atomicOr(p.status_word, (unsigned)SV_FLAG_TIMEOUT);
    }
    wr.drain(sh);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
constexpr int G_COMBOS = 3;
static std::atomic<int> g_grouped_attr[64][G_COMBOS][3];

template <typename TT, typename TD>
static constexpr int g_combo_of() {
    return std::is_same<TT, TD>::value ? (sizeof(TT) == 4 ? 0 : 1) : 2;
}

template <typename TT, typename TD, int MS>
static cudaError_t launch_grouped_ms(const VerifyParams& p, int n_cl, int cs, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    constexpr int ci = g_combo_of<TT, TD>();
    if (dev < 0 || dev >= 64 || !g_grouped_attr[dev][ci][MS - 1].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(verify_grouped_kernel<TT, TD, MS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 RING_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(verify_grouped_kernel<TT, TD, MS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) g_grouped_attr[dev][ci][MS - 1].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3((unsigned)(n_cl * cs), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)RING_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // The call may launch before the work ahead of it on the stream has
    // completed; the kernel reads no input before that work has (measured on
    // GB300, B=64 half-greedy calls one after another: 30.7 -> 30.5 us).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, verify_grouped_kernel<TT, TD, MS>, p);
}

template <typename TT, typename TD>
static cudaError_t launch_grouped_typed(const VerifyParams& p, int n_cl, int cs, cudaStream_t stream) {
    if (!p.modes && p.mode == SV_GREEDY) return launch_grouped_ms<TT, TD, MS_GREEDY>(p, n_cl, cs, stream);
    if (!p.modes && p.mode == SV_SAMPLE) return launch_grouped_ms<TT, TD, MS_SAMPLE>(p, n_cl, cs, stream);
    return launch_grouped_ms<TT, TD, MS_MIXED>(p, n_cl, cs, stream);
}

bool group_plan_fits(int B, int K, bool can_sample, int V, int esize, int n_cl, int cs) {
    if (B < 1 || B > NTHREADS || K < 0 || K > MAX_K) return false;
    if (cs < 1 || cs > G_MAX_CS || (cs & (cs - 1)) != 0) return false;
    if (n_cl < 1 || n_cl > B) return false;
    const int g_max = (B + n_cl - 1) / n_cl;
    const int rows_max = can_sample ? 2 * K + 1 : K + 1;
    if (g_max > GMAX || g_max > cs || g_max * rows_max > GROWS) return false;
    // every pass-2 group (at least cs / g_max CTAs) keeps its slice of a row
    // within the kernel's bookkeeping
    const int lo = min_cluster_size(V, esize);
    return lo > 0 && cs / g_max >= lo;
}

// Clusters of cs CTAs of the grouped kernel that fit on the GPU at once (two
// CTAs per SM, a cluster within one GPC), per device; 0 when unknown.
static std::atomic<int> g_grouped_active[64][5];

static int grouped_active_clusters(int cs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int lg = cs >= 16 ? 4 : cs >= 8 ? 3 : cs >= 4 ? 2 : cs >= 2 ? 1 : 0;
    int n = g_grouped_active[dev][lg].load(std::memory_order_acquire);
    if (n > 0) return n - 1;
    auto kernel = verify_grouped_kernel<__nv_bfloat16, __nv_bfloat16, MS_MIXED>;
    n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RING_BYTES) == cudaSuccess &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3((unsigned)cs, 1, 1);
        cfg.blockDim = dim3(NTHREADS, 1, 1);
        cfg.dynamicSmemBytes = (size_t)RING_BYTES;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    g_grouped_active[dev][lg].store(n + 1, std::memory_order_release);
    return n;
}

// Automatic plan for a lone call: clusters of 8 (else 16) CTAs, each slice
// of a row at least two pass-1 chunks; as many clusters as fit on the GPU at
// once (one wave: a cluster left for a second wave would double the call)
// while each takes at most GMAX sequences (GROWS rows); then the fewest
// clusters that keep that many sequences per cluster (so that the clusters
// hold equal counts). Used when it fills at least 80 % of two CTAs per SM;
// otherwise one cluster per sequence. (Measured on GB300, lone calls: B=64,
// K=4, V=128256 bf16, half greedy: 32 clusters of 8, 31.7 us against 37.7 us
// with one cluster of 4 per sequence. B=256, K=8, V=151936 bf16 has no such
// plan: 36 clusters of 8 fit at once, 37 are needed, and 37 took 345 us
// against 233 us.)
bool auto_group_plan(int B, int K, bool can_sample, int V, int esize, int num_sms, int& n_cl, int& cs) {
    if (B < 2 * num_sms / 16 || B > NTHREADS) return false;
    const long long nslot = ((long long)V * esize + 15) / 16;
    const int slots = 2 * num_sms;
    for (int c_try : {8, 16}) {
        if (nslot / c_try < 2 * STAGE_SLOTS) continue;
        int n = min(slots / c_try, grouped_active_clusters(c_try));
        while (n >= 1 && !group_plan_fits(B, K, can_sample, V, esize, n, c_try)) --n;
        if (n < 1) continue;
        const int g = (B + n - 1) / n;
        n = (B + g - 1) / g;
        if (n * c_try * 10 >= slots * 8 && group_plan_fits(B, K, can_sample, V, esize, n, c_try)) {
            n_cl = n;
            cs = c_try;
            return true;
        }
    }
    return false;
}

cudaError_t launch_verify_grouped(const VerifyParams& p, int dtype_target, int dtype_draft, int n_cl, int cs,
                                  cudaStream_t stream) {
    if (dtype_target == SV_F32 && dtype_draft == SV_F32) return launch_grouped_typed<float, float>(p, n_cl, cs, stream);
    if (dtype_target == SV_BF16 && dtype_draft == SV_BF16)
        return launch_grouped_typed<__nv_bfloat16, __nv_bfloat16>(p, n_cl, cs, stream);
    return cudaErrorInvalidValue;  // (fp32 target rows with bf16 draft rows come only from the LM-head path)
}

}  // namespace sv
