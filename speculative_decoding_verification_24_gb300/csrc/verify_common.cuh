// Device building blocks shared by the verify kernels over logits in HBM:
// element access, row geometry, the reductions of pass 1, the ring of
// bulk-copy stages, the draw arithmetic of pass 2 and the accept test.
// (The kernels, their shared-memory state and their launches live in
// verify_logits.cu and verify_grouped.cu.)
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "sv_device.cuh"
#include "sv_launch.h"

namespace cg = cooperative_groups;

namespace sv {

constexpr int MAX_K = 31;
constexpr int MAX_ROWS = 2 * MAX_K + 1;
constexpr unsigned FULL = 0xFFFFFFFFu;

// ---------------------------------------------------------------------------
// Debug builds (SPECVERIFY_DEBUG, built as libspecverify_debug.so): every
// global load and store of this kernel is first checked against the buffers
// of the call. A load must fall inside one of the inputs (logits, tokens,
// modes, draft counts, sequence ids, tree parents, LM-head partials), a
// store inside one of the outputs; the extents come from B, K, V and the
// element sizes. An access that does not is skipped (a load keeps its fill
// value; a bulk copy is not issued, and its stage completes empty) and sets
// SV_FLAG_DEBUG_BOUNDS in the status word. Nothing traps. Release builds
// compile every check away.
// ---------------------------------------------------------------------------
#ifdef SPECVERIFY_DEBUG
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

__device__ __forceinline__ bool dbg_within(const void* a, size_t bytes, const void* base, size_t extent) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), lo = reinterpret_cast<uintptr_t>(base);
    return base != nullptr && x >= lo && bytes <= extent && x - lo <= extent - bytes;
}

static __device__ __noinline__ bool dbg_load_ok(const VerifyParams& p, const void* a, size_t bytes) {
    const size_t B = (size_t)p.B, K1 = (size_t)p.K + 1, V = (size_t)p.V;
    const size_t tgt = B * K1 * V * (size_t)p.es_t;
    const bool ok = dbg_within(a, bytes, p.target, p.test_debug_shrink ? tgt / 2 : tgt) ||
                    dbg_within(a, bytes, p.draft, B * (K1 - 1) * V * (size_t)p.es_d) ||
                    dbg_within(a, bytes, p.tokens, B * K1 * 4) ||  // [B, K]; [B, K+1] for trees
                    dbg_within(a, bytes, p.modes, B * 4) || dbg_within(a, bytes, p.draft_lens, B * 4) ||
                    dbg_within(a, bytes, p.seq_ids, B * 8) || dbg_within(a, bytes, p.tree_parents, B * K1 * 4) ||
                    dbg_within(a, bytes, p.target_parts, (size_t)p.part_tiles * (size_t)p.part_M * 8) ||
                    dbg_within(a, bytes, p.draft_parts, (size_t)p.part_tiles * B * (K1 - 1) * 8);
    if (!ok && p.status_word) atomicOr(p.status_word, (unsigned)SV_FLAG_DEBUG_BOUNDS);
    return ok;
}

static __device__ __noinline__ bool dbg_store_ok(const VerifyParams& p, const void* a, size_t bytes) {
    const size_t B = (size_t)p.B, K1 = (size_t)p.K + 1;
    const bool ok = dbg_within(a, bytes, p.out_tokens, B * K1 * 4) || dbg_within(a, bytes, p.out_n_accepted, B * 4) ||
                    dbg_within(a, bytes, p.out_p_target, B * (K1 - 1) * 4) ||
                    dbg_within(a, bytes, p.out_p_draft, B * (K1 - 1) * 4) ||
                    dbg_within(a, bytes, p.out_residual_mass, B * 4) ||
                    dbg_within(a, bytes, p.out_draw_edges, B * 8) || dbg_within(a, bytes, p.out_last_node, B * 4);
    if (!ok && p.status_word) atomicOr(p.status_word, (unsigned)SV_FLAG_DEBUG_BOUNDS);
    return ok;
}

__device__ __forceinline__ bool load_ok(const VerifyParams& p, const void* a, size_t bytes) {
    if constexpr (kDebugBounds) return dbg_load_ok(p, a, bytes);
    return true;
}

// __ldg(a), or `fill` when a debug build finds `a` outside every input
template <typename T>
__device__ __forceinline__ T ld_in(const VerifyParams& p, const T* a, T fill) {
    if (!load_ok(p, a, sizeof(T))) return fill;
    return __ldg(a);
}

// __ldcg(a) (cached in L2 only: data another grid wrote), or `fill` as ld_in
template <typename T>
__device__ __forceinline__ T ldcg_in(const VerifyParams& p, const T* a, T fill) {
    if (!load_ok(p, a, sizeof(T))) return fill;
    return __ldcg(a);
}

// *a = v, skipped when a debug build finds `a` outside every output
template <typename T>
__device__ __forceinline__ void st_out(const VerifyParams& p, T* a, T v) {
    if constexpr (kDebugBounds) {
        if (!dbg_store_ok(p, a, sizeof(T))) return;
    }
    *a = v;
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int E = 4;                       // elements per 16-byte slot
    static constexpr int U1 = 8;                      // slots per lane per step, pass 1
    static constexpr int U2 = 4;                      // slots per lane per step, pass 2
    static constexpr uint32_t NEG_INF = 0xFF800000u;  // one -inf element word
};
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int E = 8;
    static constexpr int U1 = 8;
    static constexpr int U2 = 2;
    static constexpr uint32_t NEG_INF = 0xFF80FF80u;  // two -inf elements
};

// Element e of a 16-byte slot, widened to float.
template <typename T>
__device__ __forceinline__ float elem(const uint4& d, int e);
template <>
__device__ __forceinline__ float elem<float>(const uint4& d, int e) {
    const uint32_t w = e == 0 ? d.x : e == 1 ? d.y : e == 2 ? d.z : d.w;
    return __uint_as_float(w);
}
template <>
__device__ __forceinline__ float elem<__nv_bfloat16>(const uint4& d, int e) {
    const int k = e >> 1;
    const uint32_t w = k == 0 ? d.x : k == 1 ? d.y : k == 2 ? d.z : d.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}

// Element e (a runtime index, 0..E-1) of a 16-byte slot.
template <typename T>
__device__ __forceinline__ float elem_rt(const uint4& d, int e) {
    if constexpr (sizeof(T) == 4) {
        const uint32_t w = e == 0 ? d.x : e == 1 ? d.y : e == 2 ? d.z : d.w;
        return __uint_as_float(w);
    } else {
        const int k = e >> 1;
        const uint32_t w = k == 0 ? d.x : k == 1 ? d.y : k == 2 ? d.z : d.w;
        return (e & 1) ? bf16_hi(w) : bf16_lo(w);
    }
}

template <typename T>
__device__ __forceinline__ float load_logit(const VerifyParams& p, const T* row, int i);
template <>
__device__ __forceinline__ float load_logit<float>(const VerifyParams& p, const float* row, int i) {
    return ld_in(p, row + i, 0.0f);
}
template <>
__device__ __forceinline__ float load_logit<__nv_bfloat16>(const VerifyParams& p, const __nv_bfloat16* row, int i) {
    const unsigned short bits = ld_in(p, reinterpret_cast<const unsigned short*>(row) + i, (unsigned short)0);
    return __uint_as_float((uint32_t)bits << 16);
}

// A row seen as 16-byte slots: slot q holds elements q*E - head .. q*E - head
// + E - 1; the first and last slots may hang over the row's ends.
struct RowGeom {
    const uint4* base;
    int head;
    int nslot;
};

template <typename T>
__device__ __forceinline__ RowGeom row_geom(const T* row, int V) {
    const uintptr_t p = reinterpret_cast<uintptr_t>(row);
    const uintptr_t a = p & ~uintptr_t(15);
    RowGeom g;
    g.base = reinterpret_cast<const uint4*>(a);
    g.head = (int)((p - a) / sizeof(T));
    g.nslot = (int)((p - a + (uintptr_t)V * sizeof(T) + 15) >> 4);
    return g;
}

// Slot of row elements starting at element index i0 (which may be negative or
// run past V): elements outside [0, V) read as -inf.
template <typename T>
__device__ __forceinline__ uint4 load_partial_slot(const VerifyParams& p, const T* row, int V, int i0) {
    constexpr int E = Elem<T>::E;
    uint32_t w[4] = {Elem<T>::NEG_INF, Elem<T>::NEG_INF, Elem<T>::NEG_INF, Elem<T>::NEG_INF};
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = i0 + e;
        if (i < 0 || i >= V) continue;
        if constexpr (sizeof(T) == 4) {
            w[e] = ld_in(p, reinterpret_cast<const uint32_t*>(row) + i, Elem<T>::NEG_INF);
        } else {
            const uint32_t bits = ld_in(p, reinterpret_cast<const unsigned short*>(row) + i, (unsigned short)0xFF80u);
            const int k = e >> 1, sh = (e & 1) * 16;
            w[k] = (w[k] & ~(0xFFFFu << sh)) | (bits << sh);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__device__ __forceinline__ bool slot_full(const RowGeom& g, int V, int q) {
    constexpr int E = Elem<T>::E;
    const int i0 = q * E - g.head;
    return i0 >= 0 && i0 + E <= V;
}

template <typename T>
__device__ __forceinline__ uint4 neg_inf_slot() {
    return make_uint4(Elem<T>::NEG_INF, Elem<T>::NEG_INF, Elem<T>::NEG_INF, Elem<T>::NEG_INF);
}

// Any slot of a row, full or partial.
template <typename T>
__device__ __forceinline__ uint4 load_slot(const VerifyParams& p, const RowGeom& g, const T* row, int V, int q) {
    constexpr int E = Elem<T>::E;
    if (slot_full<T>(g, V, q)) return load_ok(p, g.base + q, 16) ? ld_stream(g.base + q) : neg_inf_slot<T>();
    return load_partial_slot<T>(p, row, V, q * E - g.head);
}

// Contiguous split of [0, n) into G parts; part g is [lo, hi). The host keeps
// n * G below 2^31 (rows of at most 2^26 slots, G <= 16).
__device__ __forceinline__ void split_range(int n, int g, int G, int& lo, int& hi) {
    lo = (int)((unsigned)n * (unsigned)g / (unsigned)G);
    hi = (int)((unsigned)n * (unsigned)(g + 1) / (unsigned)G);
}

// A warp's slots [qa, qb) of a row, split into the full interior [ia, ib) and
// the partial slots at either end (only slot 0 and the row's last slot can be
// partial), in index order: edge_lo, interior, edge_hi (-1 = none).
struct WarpSlots {
    int ia, ib, edge_lo, edge_hi;
};

template <typename T>
__device__ __forceinline__ WarpSlots warp_slots(const RowGeom& g, int V, int qa, int qb) {
    WarpSlots w{qa, qb, -1, -1};
    if (w.ia < w.ib && !slot_full<T>(g, V, w.ia)) w.edge_lo = w.ia++;
    if (w.ia < w.ib && !slot_full<T>(g, V, w.ib - 1)) w.edge_hi = --w.ib;
    return w;
}

// NaN-propagating maximum of the valid elements of U slots, as a tree (the
// dependent chain is log2 of the element count long).
template <typename T, int U>
__device__ __forceinline__ float group_max(const uint4 (&d)[U]) {
    if constexpr (sizeof(T) == 2) {
        uint32_t m[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            m[u] = max_nan_bf16x2(max_nan_bf16x2(d[u].x, d[u].y), max_nan_bf16x2(d[u].z, d[u].w));
#pragma unroll
        for (int st = 1; st < U; st *= 2)
#pragma unroll
            for (int u = 0; u + st < U; u += 2 * st) m[u] = max_nan_bf16x2(m[u], m[u + st]);
        return max_nan(bf16_lo(m[0]), bf16_hi(m[0]));
    } else {
        float m[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            m[u] = max_nan(max_nan(__uint_as_float(d[u].x), __uint_as_float(d[u].y)),
                           max_nan(__uint_as_float(d[u].z), __uint_as_float(d[u].w)));
#pragma unroll
        for (int st = 1; st < U; st *= 2)
#pragma unroll
            for (int u = 0; u + st < U; u += 2 * st) m[u] = max_nan(m[u], m[u + st]);
        return m[0];
    }
}

// NaN-propagating maximum of one slot's elements.
template <typename T>
__device__ __forceinline__ float slot_max(const uint4& d) {
    if constexpr (sizeof(T) == 2) {
        const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(d.x, d.y), max_nan_bf16x2(d.z, d.w));
        return max_nan(bf16_lo(m), bf16_hi(m));
    } else {
        return max_nan(max_nan(__uint_as_float(d.x), __uint_as_float(d.y)),
                       max_nan(__uint_as_float(d.z), __uint_as_float(d.w)));
    }
}

__device__ __forceinline__ float warp_incl_scan(float x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// ---------------------------------------------------------------------------
// Pass 1: per-lane accumulation of one group of U slots.
// ---------------------------------------------------------------------------
struct SoftAcc {
    float R;
    f32x2 a0, a1, a2, a3;  // eight running sums as four packed pairs
    bool ready;            // R is one finite value in every lane of the warp (set by the exact path)
};

__device__ __forceinline__ SoftAcc soft_acc_empty() { return SoftAcc{-INFINITY, 0ull, 0ull, 0ull, 0ull, false}; }

__device__ __forceinline__ float soft_acc_sum(const SoftAcc& a) {
    const f32x2 t = add2(add2(a.a0, a.a1), add2(a.a2, a.a3));
    float x0, x1;
    unpack2(t, x0, x1);
    return x0 + x1;
}

// The 16-byte slot as element pairs (fp32: two pairs, bf16: four pairs).
template <typename T>
__device__ __forceinline__ f32x2 slot_pair(const uint4& d, int k);
template <>
__device__ __forceinline__ f32x2 slot_pair<float>(const uint4& d, int k) {
    return k == 0 ? pack2(__uint_as_float(d.x), __uint_as_float(d.y))
                  : pack2(__uint_as_float(d.z), __uint_as_float(d.w));
}
template <>
__device__ __forceinline__ f32x2 slot_pair<__nv_bfloat16>(const uint4& d, int k) {
    const uint32_t w = k == 0 ? d.x : k == 1 ? d.y : k == 2 ? d.z : d.w;
    return bf16x2_to_f32x2(w);
}

// Adds sum 2^(l * c - R) over U slots to the running partial. R is raised to
// ceil(max * c) when the slots need it, by an exact power-of-two rescale of
// the sums; every step is a select, not a branch. A NaN maximum makes R NaN
// for good (the row is then reported invalid); an all -inf group adds zero.
template <typename T, int U>
__device__ __forceinline__ void soft_group(SoftAcc& a, const uint4 (&d)[U], float c) {
    constexpr int PAIRS = Elem<T>::E / 2;
    const float m = group_max<T, U>(d);
    const float Rn = max_nan(a.R, ceilf(m * c));
    const float sc = ex2(fmaxf(a.R - Rn, -1000.0f));  // exact 2^n; NaN (-inf - -inf) -> 0
    const f32x2 sc2 = pack2(sc, sc);
    a.a0 = mul2(a.a0, sc2);
    a.a1 = mul2(a.a1, sc2);
    a.a2 = mul2(a.a2, sc2);
    a.a3 = mul2(a.a3, sc2);
    a.R = Rn;
    const float nR = Rn == -INFINITY ? 0.0f : -Rn;
    const f32x2 c2 = pack2(c, c), nR2 = pack2(nR, nR);
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int k = 0; k < PAIRS; ++k) {
            const f32x2 e = ex2x2(fma2(slot_pair<T>(d[u], k), c2, nR2));
            switch ((u * PAIRS + k) & 3) {
                case 0: a.a0 = add2(a.a0, e); break;
                case 1: a.a1 = add2(a.a1, e); break;
                case 2: a.a2 = add2(a.a2, e); break;
                default: a.a3 = add2(a.a3, e); break;
            }
        }
    }
}

// q[u]: the slot index of d[u] for this lane (its elements start at
// q[u] * E - head).
template <typename T, int U>
__device__ __forceinline__ void arg_group(ArgPart& best, const uint4 (&d)[U], const int (&q)[U],
                                          int head) {
    constexpr int E = Elem<T>::E;
    const float m = group_max<T, U>(d);
    if (m > best.v || (m == best.v && m != -INFINITY) || (is_nan(m) && !is_nan(best.v))) {
        const bool want_nan = is_nan(m);
        int idx = INT_MAX;
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x = elem<T>(d[u], e);
                const bool hit = want_nan ? is_nan(x) : (x == m);
                const int i = q[u] * E + e - head;
                if (hit && i < idx) idx = i;
            }
        }
        if (idx != INT_MAX) best = merge_arg(best, ArgPart{m, idx});
    }
}

// Greedy accumulation of one lane over its slots in increasing index order:
// the largest slot maximum so far, that slot's index and its data. Strictly
// larger maxima replace it, so the first occurrence wins; a NaN replaces any
// number (the row is then invalid). The element index is found once, when
// the lane's partial is flushed.
struct ArgAcc {
    float v;
    int q;
    uint4 d;
};

__device__ __forceinline__ ArgAcc arg_acc_empty() { return ArgAcc{-INFINITY, -1, make_uint4(0u, 0u, 0u, 0u)}; }

template <typename T, int U>
__device__ __forceinline__ void arg_slots(ArgAcc& a, const uint4 (&d)[U], const int (&q)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float m = slot_max<T>(d[u]);
        const bool take = m > a.v || (is_nan(m) && !is_nan(a.v));
        if (take) {
            a.v = m;
            a.q = q[u];
            a.d = d[u];
        }
    }
}

// The lane's (value, lowest element index) from its accumulation.
template <typename T>
__device__ __forceinline__ ArgPart arg_acc_part(const ArgAcc& a, int head) {
    constexpr int E = Elem<T>::E;
    int idx = INT_MAX;
    if (a.q >= 0) {
        const bool want_nan = is_nan(a.v);
#pragma unroll
        for (int e = E - 1; e >= 0; --e) {
            const float x = elem<T>(a.d, e);
            if (want_nan ? is_nan(x) : x == a.v) idx = a.q * E + e - head;
        }
    }
    return ArgPart{a.v, idx};
}

// ---------------------------------------------------------------------------
// Ring, row table and chunk schedule.
// ---------------------------------------------------------------------------
constexpr int NCW = 8;                          // warps per CTA; each streams its own chunks
constexpr int NTHREADS = NCW * 32;
constexpr int STAGE_BYTES = 4096;               // one ring stage
constexpr int NBUF = 3;                         // stages per warp
constexpr int NSTAGE = NBUF * NCW;              // warp w owns stages w, w + NCW, w + 2 NCW
constexpr int RING_BYTES = STAGE_BYTES * NSTAGE;
constexpr int STAGE_SLOTS = STAGE_BYTES / 16;   // slots per pass-1 chunk (256)
constexpr int P2_SLOTS = STAGE_SLOTS / 2;       // target slots per pass-2 chunk (128)
constexpr int P2_DRAFT_OFF = P2_SLOTS * 16;     // draft half of a pass-2 stage
constexpr int MAX_P2_CHUNKS = 256;              // per CTA slice of one row
constexpr int MAX_CS = 16;
constexpr int MAX_ORDERED_B = 256;              // batches up to this size are taken sample-first
constexpr uint32_t WAIT_LIMIT = 1u << 22;       // polls before a wait gives up

// One row of the sequence as this CTA sees it: the 16-byte slots of its slice,
// split into the full interior [ia, ib) and the partial end slots. The pass-1
// schedule cuts every row's interior into chunks of STAGE_SLOTS slots (the
// last one of a row may be shorter) and numbers them row after row: row r
// owns chunks [c1 of row r - 1 (0 for row 0), c1), its k-th chunk holding
// slots ia + k * STAGE_SLOTS ...
struct RowInfo {
    const uint4* base;  // 16-byte aligned address of slot 0
    int head;           // elements between base and the row's first element
    int ia, ib, edge_lo, edge_hi;
    int c1;
};

__device__ __forceinline__ int row_c0(const RowInfo* rows, int r) { return r == 0 ? 0 : rows[r - 1].c1; }

// Target row i and draft row i of sequence b in the [B, K+1, V] and [B, K, V]
// layouts. A sequence verifying Kb <= K drafts reads its rows 0..Kb and
// 0..Kb-1; its row table numbers them 0..Kb (target) then Kb+1..2Kb (draft).
template <typename TT>
__device__ __forceinline__ const TT* target_row(const TT* tgt, int b, int K, int V, int i) {
    return tgt + ((size_t)b * (K + 1) + i) * V;
}
template <typename TD>
__device__ __forceinline__ const TD* draft_row(const TD* drf, int b, int K, int V, int i) {
    return drf + ((size_t)b * K + i) * V;
}

// E_TT consecutive elements of a TD row starting at element i0, in the slot
// format of TT (elements outside [0, V) read as -inf). The mixed case widens
// bf16 draft elements exactly into fp32 words.
template <typename TT, typename TD>
__device__ __forceinline__ uint4 load_elems_as(const VerifyParams& p, const TD* row, int V, int i0) {
    if constexpr (std::is_same<TT, TD>::value) {
        return load_partial_slot<TT>(p, row, V, i0);
    } else {
        static_assert(sizeof(TT) == 4 && sizeof(TD) == 2, "mixed rows: fp32 target, bf16 draft");
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = i0 + e;
            w[e] = (i >= 0 && i < V)
                       ? ((uint32_t)ld_in(p, reinterpret_cast<const unsigned short*>(row) + i, (unsigned short)0xFF80u) << 16)
                       : 0xFF800000u;
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <typename T>
__device__ __forceinline__ RowInfo make_row_info(const T* row, int V, int rank, int CS) {
    const RowGeom g = row_geom(row, V);
    int qa, qb;
    split_range(g.nslot, rank, CS, qa, qb);
    const WarpSlots sl = warp_slots<T>(g, V, qa, qb);
    return RowInfo{g.base, g.head, sl.ia, sl.ib, sl.edge_lo, sl.edge_hi, 0};
}

struct DrawRows {
    float c;
    float ntR, invSt;   // target row j: -R and 1/S
    float ndR, invSd;   // draft row j (use_d only)
    bool use_d;
    f32x2 c2, ntR2, invSt2, ndR2, invSd2;  // the same, packed for fp32x2 arithmetic
};

__device__ __forceinline__ void pack_draw_rows(DrawRows& w) {
    w.c2 = pack2(w.c, w.c);
    w.ntR2 = pack2(w.ntR, w.ntR);
    w.invSt2 = pack2(w.invSt, w.invSt);
    w.ndR2 = pack2(w.ndR, w.ndR);
    w.invSd2 = pack2(w.invSd, w.invSd);
}

// The draw mass of an element pair, bit-identical to draw_mass on each half.
__device__ __forceinline__ f32x2 draw_mass2(const DrawRows& w, f32x2 lt, f32x2 ld) {
    const f32x2 pt = mul2(ex2x2(fma2(lt, w.c2, w.ntR2)), w.invSt2);
    if (!w.use_d) return pt;
    const f32x2 pd = mul2(ex2x2(fma2(ld, w.c2, w.ndR2)), w.invSd2);
    float a, b;
    unpack2(fma2(pd, pack2(-1.0f, -1.0f), pt), a, b);  // pt - pd, rounded once
    return pack2(fmaxf(a, 0.0f), fmaxf(b, 0.0f));
}

__device__ __forceinline__ float draw_mass(const DrawRows& w, float lt, float ld) {
    const float pt = ex2(fmaf(lt, w.c, w.ntR)) * w.invSt;
    if (!w.use_d) return pt;
    const float pd = ex2(fmaf(ld, w.c, w.ndR)) * w.invSd;
    return fmaxf(pt - pd, 0.0f);
}

template <typename T>
__device__ __forceinline__ float slot_mass(const DrawRows& w, const uint4& dt, const uint4& dd) {
    constexpr int E = Elem<T>::E;
    float ls = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ls += draw_mass(w, elem<T>(dt, e), elem<T>(dd, e));
    return ls;
}

// The rows of the final draw: target row j and (use_d) draft row j. The
// draft shares the target's 16-byte slots only when both have the same type
// and alignment; otherwise its elements are read one by one.
template <typename TT, typename TD>
struct DrawSrc {
    const TT* trow;
    const TD* drow;
    RowGeom gt, gd;
    int V;
    bool same_slots;
};

// Target slot q (target geometry) and the draft elements with the same
// indices, from global memory; q < 0 gives empty slots.
template <typename TT, typename TD>
__device__ __forceinline__ void load_draw_slot(const VerifyParams& p, const DrawSrc<TT, TD>& src, bool use_d, int q,
                                               uint4& dt, uint4& dd) {
    constexpr int E = Elem<TT>::E;
    if (q < 0) {
        dt = neg_inf_slot<TT>();
        dd = neg_inf_slot<TT>();
        return;
    }
    dt = load_slot<TT>(p, src.gt, src.trow, src.V, q);
    if (!use_d) dd = neg_inf_slot<TT>();
    else if (src.same_slots) dd = load_slot<TT>(p, src.gd, reinterpret_cast<const TT*>(src.drow), src.V, q);
    else dd = load_elems_as<TT, TD>(p, src.drow, src.V, q * E - src.gt.head);
}

// One 32-slot step of the final search, for the warp that owns it: lane l
// holds slot q_begin + step * 32 + l of the part (valid below n). Each
// element's draw mass is formed once; the lane keeps them, with the warp's
// inclusive scan of the slot sums in the pass-2 order.
template <typename TT, typename TD>
struct DrawStep {
    static constexpr int E = Elem<TT>::E;
    float m[E];        // this lane's element masses
    float incl, prev;  // inclusive scan of the slot sums: this lane and lane - 1
    float tot;         // the step's total
    int last_pos;      // the warp's last element with positive mass (-1: none)
    int i0;            // row element index of this lane's first element

    __device__ __forceinline__ void load(const VerifyParams& p, const DrawSrc<TT, TD>& src, const DrawRows& w,
                                         int q_begin, int n, int step, int lane) {
        const int i = step * 32 + lane;
        const int q = i < n ? q_begin + i : -1;
        uint4 dt, dd;
        load_draw_slot<TT, TD>(p, src, w.use_d, q, dt, dd);
        take(w, dt, dd, q, src.gt.head, lane);
    }

    // The same from slots already at hand: target slot q (q < 0: none) and
    // the draft elements with the same indices, in the target's slot format.
    __device__ __forceinline__ void take(const DrawRows& w, const uint4& dt, const uint4& dd, int q, int head,
                                         int lane) {
        i0 = q * E - head;
        float ls = 0.0f;
        int lp = -1;
#pragma unroll
        for (int k2 = 0; k2 < E / 2; ++k2) {
            unpack2(draw_mass2(w, slot_pair<TT>(dt, k2), slot_pair<TT>(dd, k2)), m[2 * k2], m[2 * k2 + 1]);
            ls += m[2 * k2];
            ls += m[2 * k2 + 1];
        }
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (q >= 0 && m[e] > 0.0f) lp = i0 + e;
        incl = warp_incl_scan(ls, lane);
        prev = __shfl_up_sync(FULL, incl, 1);
        tot = __shfl_sync(FULL, incl, 31);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(FULL, lp, o));
        last_pos = lp;
    }

    // The element of lane l's slot where the cumulative mass from `run`
    // (the masses before this lane) first exceeds tw; its last positive
    // element if rounding leaves tw past it. d0, d1: tw's distances to the
    // chosen element's lower and upper cumulative edges (0, 0 in the
    // rounding case).
    __device__ __forceinline__ int walk(ff run, ff tw, int l, float& d0, float& d1) const {
        ff cum = ff_add(run, l == 0 ? 0.0f : prev);
        int tok = -1, lastp = -1;
        d0 = 0.0f;
        d1 = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (m[e] > 0.0f) {
                lastp = i0 + e;
                const ff below = cum;
                cum = ff_add(cum, m[e]);
                if (tok < 0 && ff_gt(cum, tw)) {
                    tok = i0 + e;
                    const ff a = ff_add(tw, ff_neg(below)), z = ff_add(cum, ff_neg(tw));
                    d0 = a.hi + a.lo;
                    d1 = z.hi + z.lo;
                }
            }
        }
        return tok < 0 ? lastp : tok;
    }
};

// The accept test u * P_d(x) < P_t(x) with P = e / S, i.e. u * e_d * S_t <
// e_t * S_d, decided as if in exact arithmetic on these float inputs. The
// float products carry relative errors below 2^-23 (left, two roundings) and
// 2^-24 (right) while they stay far above the float underflow range; outside
// a 2^-21 band around equality they decide it, inside it (or near underflow)
// the products are formed in double, where u * e_d and e_t * S_d are exact.
static __device__ __noinline__ bool accept_draft_exact(float u, float ed, float St, float et, float Sd) {
    return (double)u * (double)ed * (double)St < (double)et * (double)Sd;
}

__device__ __forceinline__ bool accept_draft(float u, float ed, float St, float et, float Sd) {
    const float ue = u * ed;
    const float l = ue * St, r = et * Sd;
    const float tiny = 0x1p-100f;
    const bool normal = ue >= tiny && l >= tiny && r >= tiny;
    const bool sure_accept = normal && l < r * (1.0f - 0x1p-21f);
    const bool sure_reject = normal && l > r * (1.0f + 0x1p-21f);
    if (sure_accept) return true;
    if (sure_reject) return false;
    return accept_draft_exact(u, ed, St, et, Sd);
}

// The NBUF ring stages a warp owns (w, w + NCW, ...). Chunk number `seq` of
// this warp (counted over both passes) lives in stage seq % NBUF and is that
// stage's (seq / NBUF)-th fill, so its mbarrier phase parity is
// (seq / NBUF) & 1. Fills are issued in seq order; `filled` and `waited`
// count them. The warp refills a stage itself once it has copied the stage
// into registers.
struct WarpRing {
    int warp;
    uint32_t filled, waited;
    template <class SH>
    __device__ __forceinline__ uint64_t* bar(SH& sh, uint32_t seq) const {
        return &sh.full[warp + NCW * (int)(seq % NBUF)];
    }
    __device__ __forceinline__ char* stage(char* ring, uint32_t seq) const {
        return ring + (warp + NCW * (int)(seq % NBUF)) * STAGE_BYTES;
    }
    // Lane 0 announces the bytes of fill `seq`; its copies follow (also lane 0).
    template <class SH>
    __device__ __forceinline__ void begin_fill(SH& sh, uint32_t seq, uint32_t bytes, int lane) {
        if (lane == 0) mbar_arrive_expect_tx(bar(sh, seq), bytes);
        filled = seq + 1;
    }
    template <class SH>
    __device__ __forceinline__ bool wait(SH& sh, uint32_t seq) {
        waited = seq + 1;
        return mbar_wait(bar(sh, seq), (seq / NBUF) & 1, WAIT_LIMIT);
    }
    // Before the CTA exits: every copy this warp issued has landed (bounded).
    template <class SH>
    __device__ __forceinline__ void drain(SH& sh) {
        for (uint32_t q = waited; q < filled; ++q) (void)mbar_wait(bar(sh, q), (q / NBUF) & 1, WAIT_LIMIT);
        waited = filled;
    }
};

template <typename T, bool SAMPLE, class SH>
__device__ __forceinline__ void flush_row(SH& sh, int warp, int lane, int row,
                                          const SoftAcc& sa, const ArgAcc& aa, int head) {
    if (SAMPLE) {
        SoftPart pp{sa.R, soft_acc_sum(sa)};
        if (sa.R == -INFINITY) pp.s = 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            pp = merge_soft(pp, SoftPart{__shfl_xor_sync(FULL, pp.R, o), __shfl_xor_sync(FULL, pp.s, o)});
        if (lane == 0) sh.warp_part[warp][row] = pack(pp);
    } else {
        ArgPart ag = arg_acc_part<T>(aa, head);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ag = merge_arg(ag, ArgPart{__shfl_xor_sync(FULL, ag.v, o), __shfl_xor_sync(FULL, ag.i, o)});
        if (lane == 0) sh.warp_part[warp][row] = pack(ag);
    }
}

constexpr int CHUNK_LANE_SLOTS = STAGE_SLOTS / 32;  // 8 slots per lane

// A chunk of one row held by a lane: slot u of d is chunk slot u * 32 + lane,
// valid below n; q0 is the row slot of chunk slot 0. Reduced in groups of
// GROUP_SLOTS slots per lane.
constexpr int GROUP_SLOTS = 4;

// Limit of a lane's chunk sum on the fast path: below it, no element of the
// chunk exceeds the lane's R by more than log2(FAST_SUM_LIMIT) = 12 (in units
// of l * c), so every later sum and product of the step stays far from the
// float32 range's end.
constexpr float FAST_SUM_LIMIT = 4096.0f;

// Fast path of a full chunk in sample mode: 2^(l * c - R) at the lane's
// current R, with no per-group maximum and no rescale, summed into
// chunk-local pairs. Returns false (and leaves the running partial as it
// was) when the chunk needs the exact path: a lane without a finite R yet,
// or a lane sum of FAST_SUM_LIMIT or more, infinite or NaN (an element well
// above R, +inf or NaN). The decision is warp-uniform.
template <typename T>
__device__ __forceinline__ bool soft_chunk_fast(SoftAcc& sa, const uint4 (&d)[CHUNK_LANE_SLOTS], float c) {
    constexpr int PAIRS = Elem<T>::E / 2;
    if (!sa.ready) return false;
    const f32x2 c2 = pack2(c, c), nR2 = pack2(-sa.R, -sa.R);
    f32x2 b0 = 0ull, b1 = 0ull, b2 = 0ull, b3 = 0ull;
#pragma unroll
    for (int u = 0; u < CHUNK_LANE_SLOTS; ++u) {
#pragma unroll
        for (int k = 0; k < PAIRS; ++k) {
            const f32x2 e = ex2x2(fma2(slot_pair<T>(d[u], k), c2, nR2));
            switch ((u * PAIRS + k) & 3) {
                case 0: b0 = add2(b0, e); break;
                case 1: b1 = add2(b1, e); break;
                case 2: b2 = add2(b2, e); break;
                default: b3 = add2(b3, e); break;
            }
        }
    }
    float x0, x1;
    unpack2(add2(add2(b0, b1), add2(b2, b3)), x0, x1);
    if (__any_sync(FULL, !(x0 + x1 < FAST_SUM_LIMIT))) return false;
    sa.a0 = add2(sa.a0, b0);
    sa.a1 = add2(sa.a1, b1);
    sa.a2 = add2(sa.a2, b2);
    sa.a3 = add2(sa.a3, b3);
    return true;
}

template <typename T, bool SAMPLE>
__device__ __forceinline__ void reduce_chunk(SoftAcc& sa, ArgAcc& aa, const uint4 (&d)[CHUNK_LANE_SLOTS],
                                             int n, int q0, float c, int lane) {
    const bool whole = n == STAGE_SLOTS;
    if (SAMPLE && whole && soft_chunk_fast<T>(sa, d, c)) return;
    // (slots past the end of a partial chunk were loaded as -inf)
#pragma unroll
    for (int g = 0; g < CHUNK_LANE_SLOTS / GROUP_SLOTS; ++g) {
        uint4 x[GROUP_SLOTS];
        int qs[GROUP_SLOTS];
#pragma unroll
        for (int u = 0; u < GROUP_SLOTS; ++u) {
            const int i = (g * GROUP_SLOTS + u) * 32 + lane;
            x[u] = d[g * GROUP_SLOTS + u];
            qs[u] = q0 + i;
        }
        if (SAMPLE) soft_group<T, GROUP_SLOTS>(sa, x, c);
        else arg_slots<T, GROUP_SLOTS>(aa, x, qs);
    }
    if (SAMPLE) {
        // One R for the whole warp (its lanes' maximum, NaN-propagating; an
        // exact power-of-two rescale of each lane's sums), so that the fast
        // path of the next chunks falls back only when an element exceeds
        // the largest one the warp has seen by 2^12.
        float Rw = sa.R;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Rw = max_nan(Rw, __shfl_xor_sync(FULL, Rw, o));
        const float sc = sa.R == -INFINITY ? 0.0f : ex2(fmaxf(sa.R - Rw, -1000.0f));
        const f32x2 sc2 = pack2(sc, sc);
        sa.a0 = mul2(sa.a0, sc2);
        sa.a1 = mul2(sa.a1, sc2);
        sa.a2 = mul2(sa.a2, sc2);
        sa.a3 = mul2(sa.a3, sc2);
        sa.R = Rw;
        sa.ready = Rw > -INFINITY && Rw < INFINITY;
    }
}

// The row of pass-1 chunk `chunk` for a warp that visits chunks in order.
struct RowCursor {
    int r, c0, c1;
};

// The refill cursor, with its row's geometry in registers (looked up once a row).
struct FillCursor {
    RowCursor rc;
    const uint4* base;
    int ia, ib;
};

__device__ __forceinline__ void seek_row(RowCursor& rc, const RowInfo* rows, int chunk) {
    while (chunk >= rc.c1) {  // rows with no chunk of their own are skipped
        ++rc.r;
        rc.c0 = rc.c1;
        rc.c1 = rows[rc.r].c1;
    }
}

// Issues the bulk copy of pass-1 chunk `chunk` (one piece of one row) as fill
// `fseq` of the warp; lane 0 issues.
template <class SH>
__device__ __forceinline__ void fill_pass1(const VerifyParams& p, SH& sh, WarpRing& wr, char* ring,
                                           uint32_t fseq, int chunk, FillCursor& fc, int lane) {
    if (chunk >= fc.rc.c1) {
        seek_row(fc.rc, sh.rows, chunk);
        const RowInfo& ri = sh.rows[fc.rc.r];
        fc.base = ri.base;
        fc.ia = ri.ia;
        fc.ib = ri.ib;
    }
    const int q0 = fc.ia + (chunk - fc.rc.c0) * STAGE_SLOTS;
    const int n = min(STAGE_SLOTS, fc.ib - q0);
    // (a debug build that finds the copy out of bounds completes the stage empty)
    const bool ok = lane != 0 || load_ok(p, fc.base + q0, (size_t)n * 16u);
    wr.begin_fill(sh, fseq, ok ? (uint32_t)n * 16u : 0u, lane);
    if (lane == 0 && ok)
        bulk_g2s_hint(wr.stage(ring, fseq), fc.base + q0, (uint32_t)n * 16u, wr.bar(sh, fseq), l2_evict_first_policy());
}

// The 16-byte aligned span of a bf16 draft row that holds the elements of
// fp32 target slots [q, q + n) (interior slots: every element lies in
// [0, V), so the span stays inside the 16-byte blocks of the row's own
// elements); `off` is the first element's byte offset in the span.
struct DraftSpan {
    const char* base;
    uint32_t bytes, off;
};
template <typename TT, typename TD>
__device__ __forceinline__ DraftSpan draft_span(const DrawSrc<TT, TD>& src, int q, int n) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src.drow) + 2 * (uintptr_t)(q * 4 - src.gt.head);
    const uintptr_t a0 = s0 & ~(uintptr_t)15, a1 = (s0 + 8 * (uintptr_t)n + 15) & ~(uintptr_t)15;
    return DraftSpan{reinterpret_cast<const char*>(a0), (uint32_t)(a1 - a0), (uint32_t)(s0 - a0)};
}

// Draft elements of target slot i of a pass-2 chunk, from its span in the
// stage, widened exactly into an fp32 slot.
__device__ __forceinline__ uint4 span_slot(const char* span, uint32_t off, int i) {
    const char* p = span + off + 8 * i;
    uint32_t w0, w1;
    if ((off & 7u) == 0) {
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(smem_u32(p)));
    } else {
        unsigned short h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h[k]) : "r"(smem_u32(p + 2 * k)));
        w0 = (uint32_t)h[0] | ((uint32_t)h[1] << 16);
        w1 = (uint32_t)h[2] | ((uint32_t)h[3] << 16);
    }
    return make_uint4(w0 << 16, w0 & 0xFFFF0000u, w1 << 16, w1 & 0xFFFF0000u);
}

// Issues pass-2 chunk ci (target slots, and the draft slots when they share
// the target's alignment, or the draft's span of them when the draft is bf16
// under an fp32 target) as fill `fseq` of the warp.
template <typename TT, typename TD, class SH>
__device__ __forceinline__ void fill_pass2(const VerifyParams& p, SH& sh, WarpRing& wr, char* ring,
                                           uint32_t fseq, const DrawSrc<TT, TD>& src, int ia, int ib, int ci,
                                           bool ring_d, bool span_d, int lane) {
    const int q = ia + ci * P2_SLOTS;
    const int n = min(P2_SLOTS, ib - q);
    const DraftSpan ds = span_d ? draft_span<TT, TD>(src, q, n) : DraftSpan{nullptr, 0u, 0u};
    // (a debug build issues only the copies it finds in bounds, and expects their bytes)
    const bool ok_t = lane != 0 || load_ok(p, src.gt.base + q, (size_t)n * 16u);
    const bool ok_d = !ring_d || lane != 0 || load_ok(p, src.gd.base + q, (size_t)n * 16u);
    const bool ok_s = !span_d || lane != 0 || load_ok(p, ds.base, ds.bytes);
    wr.begin_fill(sh, fseq,
                  (ok_t ? (uint32_t)n * 16u : 0u) + (ring_d && ok_d ? (uint32_t)n * 16u : 0u) + (ok_s ? ds.bytes : 0u),
                  lane);
    if (lane == 0) {
        char* stage = wr.stage(ring, fseq);
        if (ok_t) bulk_g2s(stage, src.gt.base + q, (uint32_t)n * 16u, wr.bar(sh, fseq));
        if (ring_d && ok_d) bulk_g2s(stage + P2_DRAFT_OFF, src.gd.base + q, (uint32_t)n * 16u, wr.bar(sh, fseq));
        if (span_d && ok_s) bulk_g2s(stage + P2_DRAFT_OFF, ds.base, ds.bytes, wr.bar(sh, fseq));
    }
}

// The rules a launch can meet: sample only, greedy only (also trees), or both
// (per-sequence modes). Each set is its own instantiation, so a uniform batch
// runs a kernel without the other rule's code (fewer instructions to fetch in
// the phases that run once per call).
constexpr int MS_SAMPLE = 1, MS_GREEDY = 2, MS_MIXED = 3;

}  // namespace sv
