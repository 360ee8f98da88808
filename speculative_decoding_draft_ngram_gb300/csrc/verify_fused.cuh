// spec_verify in one persistent kernel (sm_103a): the streaming pass and the
// decisions of the sequences run side by side, so a sequence is decided as
// soon as the rows it needs have been streamed instead of after the whole
// batch.  Included by verify.cuh (it uses that file's helpers).
//
// Method: SwiftLM page, paragraph on algorithmic equivalence after Leviathan
// et al. (accept with P_target / P_draft, resample from the corrected
// distribution on rejection, bonus token when all drafts are accepted); AX
// Engine page, "Core Technical Architecture & Methods" (EMA gate, rollback
// by moving the sequence-length pointer).
//
// One CTA per SM, 20 warps:
//   * warp 16, the producer: walks this CTA's share of the call's row-chunks
//     and keeps up to kStages of them in flight with cp.async.bulk into a
//     shared-memory ring (as in the streaming kernel of the two-kernel
//     schedule).  The rows are ordered row index first -- every active
//     sequence's row 0, then every row 1, ... -- and dealt out round robin
//     (row t to CTA t mod G), so at any moment all CTAs work near the same
//     point of that order, a sequence's rows complete one after the other
//     during the call, and the CTA that streams a row also decides it.
//   * warps 0..15 stream each chunk: per noise block the bound of its
//     sampling scores (T > 0; the block draws come from the producer) or its
//     largest raw logit (T = 0), and for the rows that carry an accept test
//     the sum of exponentials of the chunk.  The warp that finishes a row's
//     last chunk hands the row to the decision group (shared-memory ring).
//   * warps 17..19, the decision group: for each row it streamed, the accept
//     test of d_{j+1} (T > 0; the normaliser from the chunk sums) or the
//     row's argmax (T = 0).  The outcome is or-ed into the sequence's state
//     word (global, tagged with the call's epoch); the one update that makes
//     a = (number accepted before the first rejection) known -- a rejection
//     at row a with rows 0..a-1 accepted, or all k_eff drafts accepted and
//     row k_eff streamed -- samples the token at row a (whichever CTA
//     streamed it) and writes the sequence's outputs.
//   * early exit (optional): the producer skips the chunks of rows past a
//     sequence's known first rejection; they cannot change the outputs.
//   * the last CTA to finish (a grid ticket) writes the EMAs and the cooling
//     counts: every CTA reads them at its start to plan the work, so none may
//     change before all have finished.
// No CTA ever waits for another: the cross-CTA steps are tickets.  Every
// wait inside a CTA (ring barriers, the note ring, the group's poll) is
// bounded and raises TIMEOUT when it gives up.
#pragma once

namespace specng {

constexpr int kFDWarps = 3;                                  // decision group
constexpr int kFD0 = kCWarps + 1;                            // its first warp
constexpr int kFThreads = (kCWarps + 1 + kFDWarps) * 32;     // 640
constexpr int kFDThreads = kFDWarps * 32;
constexpr int kFusedMaxB = 2048;                             // sequences per call on this schedule
constexpr int kNoteCap = 256;                                // streamed rows waiting for the decision group
constexpr int kStateAcc = SPECNG_MAX_K + 1;                  // accept bits start here
constexpr int kStateEpoch = 2 * SPECNG_MAX_K + 1;            // epoch bits start here
constexpr unsigned long long kStateBits = (1ull << kStateEpoch) - 1ull;
static_assert(kStateEpoch + 31 == 64, "state word layout");

template <bool BF16> __host__ __device__ constexpr int fused_batch() { return BF16 ? 4 : 2; }
template <bool BF16> __host__ __device__ constexpr int fused_vpl() { return BF16 ? 1 : 2; }
template <bool BF16>
__host__ __device__ constexpr size_t fused_stage_bytes() {
    return static_cast<size_t>(kFDWarps) * fused_batch<BF16>() * 32 * fused_vpl<BF16>() * 16;
}
template <bool BF16, bool PENALTY>
__host__ __device__ constexpr size_t fused_dyn_smem() {
    return static_cast<size_t>(kStages) * kChunkBytes + (PENALTY ? static_cast<size_t>(kStages) * (kChunkBytes / 16) : 0) +
           fused_stage_bytes<BF16>() + static_cast<size_t>(kFusedMaxB) * 3 +
           (PENALTY ? static_cast<size_t>(2 * kPenSlots) * 4 : 0);
}

__device__ __forceinline__ void group_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kFDThreads) : "memory"); }

// Accept length a known from a state word (bits of this call), or -1.
__device__ __forceinline__ int known_a(unsigned long long st, int keff) {
    for (int j = 0; j <= keff; ++j) {
        if (!((st >> j) & 1ull)) return -1;
        if (j == keff) return keff;
        if (!((st >> (kStateAcc + j)) & 1ull)) return j;
    }
    return -1;
}

__device__ __forceinline__ unsigned long long state_bits(unsigned long long w, uint32_t epoch) {
    return (w >> kStateEpoch) == epoch ? (w & kStateBits) : 0ull;
}

// Or bits into a sequence's state word (words of an older call count as
// empty).  Returns the bits before the update, or ~0 when the bounded
// retry loop gave up.
__device__ __forceinline__ unsigned long long state_or(unsigned long long* p, uint32_t epoch, unsigned long long bits) {
    unsigned long long old = __ldcg(p);
    for (int it = 0; it < (1 << 16); ++it) {
        const unsigned long long cur = state_bits(old, epoch);
        const unsigned long long nv = (static_cast<unsigned long long>(epoch) << kStateEpoch) | cur | bits;
        const unsigned long long prev = atomicCAS(p, old, nv);
        if (prev == old) return cur;
        old = prev;
    }
    return ~0ull;
}

// Shared state of the decision group.
struct DShared {
    double red[kFDWarps];
    Top2 top[kFDWarps];
    unsigned thr;
    int ival[4];
    int d[SPECNG_MAX_K + 1];
    int rows[32];
    int nrows;
    int quit;
    int nh;
    unsigned pmask[kFDWarps][16];
};

// Is v among the last W tokens of history[:L] ++ d_1..d_j (the penalty window
// of row j of sequence b)?  One whole warp; S.d holds the drafts.
__device__ __forceinline__ bool warp_window_has(const VerifyDev& P, const DShared& S, int b, int j, int v) {
    int L = P.lens[b];
    L = L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
    const int nh = L < P.W ? L : P.W;
    const int total = nh + j;
    const int cnt = total < P.W ? total : P.W;
    const int* tail = P.hist + static_cast<size_t>(b) * P.hist_stride + (L - nh);
    bool f = false;
    for (int t = (threadIdx.x & 31); t < cnt; t += 32) {
        const int idx = total - cnt + t;
        f |= (idx < nh ? tail[idx] : S.d[idx - nh]) == v;
    }
    return __any_sync(0xffffffffu, f);
}

// With the penalty: sequence b's history tail into the window table (token ->
// latest position in the tail), for the per-element lookups of a sampling or
// an argmax.  Whole group; S.d holds the drafts.
template <bool PENALTY>
__device__ __forceinline__ void group_load_seq(const VerifyDev& P, DShared& S, int* pkey, int* ppos, int b, int gt) {
    if constexpr (PENALTY) {
        int L = P.lens[b];
        L = L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
        const int nh = L < P.W ? L : P.W;
        for (int t = gt; t < kPenSlots; t += kFDThreads) {
            pkey[t] = -1;
            ppos[t] = -1;
        }
        if (gt == 0) S.nh = nh;
        group_sync();
        const int* tail = P.hist + static_cast<size_t>(b) * P.hist_stride + (L - nh);
        for (int t = gt; t < nh; t += kFDThreads) {
            const int v = tail[t];
            if (v < 0) continue;
            uint32_t h = pen_hash(v);
            for (int probe = 0; probe < kPenSlots; ++probe) {
                const int old = atomicCAS(&pkey[h], -1, v);
                if (old == -1 || old == v) {
                    atomicMax(&ppos[h], t);
                    break;
                }
                h = (h + 1u) & (kPenSlots - 1u);
            }
        }
    } else {
        if (gt == 0) S.nh = 0;
        group_sync();
    }
}

// The normaliser of a row from its chunks' segment sums (one warp): the
// largest reference and the sum relative to it.
__device__ __forceinline__ void row_normaliser(const VerifyDev& P, size_t row, int lane, float& mf, float& Sf) {
    const SegSum* pr = P.part + row * P.nchunk;
    mf = -INFINITY;
    for (int c = lane; c < P.nchunk; c += 32) mf = fmaxf(mf, __ldcg(&pr[c].m));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mf = fmaxf(mf, __shfl_xor_sync(0xffffffffu, mf, off));
    Sf = 0.0f;
    for (int c = lane; c < P.nchunk; c += 32) {
        const float2 p = __ldcg(reinterpret_cast<const float2*>(pr + c));
        if (p.x > -INFINITY) Sf += p.y * ex2_approx((p.x - mf) * P.sc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Sf += __shfl_xor_sync(0xffffffffu, Sf, off);
}

// Argmax of transformed row j of sequence b (T = 0), lowest id on ties: the
// block with the largest raw value first, then every block whose bound is
// within the tie margin of the best.  Whole group; returns the winner.
template <bool BF16, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ int group_argmax(const VerifyDev& P, DShared& S, const int* pkey, const int* ppos, int b, int j) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int BLK = 1 << kNoiseBlockShift;
    constexpr int VPL = fused_vpl<BF16>();
    const int gt = threadIdx.x - kFD0 * 32, gw = gt >> 5, lane = gt & 31;
    const size_t row = static_cast<size_t>(b) * (P.K + 1) + j;
    const float* bmx = P.bmax + row * P.nblk;
    const char* rowp = static_cast<const char*>(P.logits) + row * P.V * ElemTraits<BF16>::SIZE;
    auto pen_of = [&](int v) { return PENALTY && pen_lookup(pkey, ppos, S.d, S.nh, P.W, v, j); };
    Top2 t = top2_empty();
    auto scan = [&](int q, float gth) {
        uint4 r[VPL];
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int e0 = q * BLK + (u * 32 + lane) * EPV;
            r[u] = e0 < P.V ? load_vec_chk<BF16>(P, rowp, e0, P.V) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            float x[EPV];
            unpack<BF16>(r[u], x);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const int v = q * BLK + (u * 32 + lane) * EPV + e;
                if (v >= P.V) continue;
                const float z = transform_f32<SOFTCAP, PENALTY>(x[e], pen_of(v), P);
                if (z >= gth) top2_push(t, z, v);
            }
        }
    };
    if (gt == 0) S.thr = 0u;
    group_sync();
    // seed: the largest transformed value in this warp's block with the largest raw
    // value (blocks q = gw mod kFDWarps) sets the tie threshold; nothing is kept, so
    // the pass below meets every element once
    {
        float lb = -INFINITY;
        int lq = -1;
        for (int q = gw + kFDWarps * lane; q < P.nblk; q += kFDThreads) {
            const float x = __ldcg(bmx + q);
            if (lq < 0 || x > lb) { lb = x; lq = q; }
        }
        const unsigned kq = __reduce_max_sync(0xffffffffu, lq >= 0 ? score_key(lb) | 1u : 0u);
        const unsigned own = __ballot_sync(0xffffffffu, lq >= 0 && (score_key(lb) | 1u) == kq);
        const int q0 = own ? __shfl_sync(0xffffffffu, lq, __ffs(own) - 1) : -1;
        float zb = -INFINITY;
        if (q0 >= 0) {
            scan(q0, -INFINITY);  // t is empty before: keep only its best value
            zb = t.s1;
            t = top2_empty();
        }
        const unsigned kw = warp_best_key(zb);
        if (kw != 0u && lane == 0) atomicMax(&S.thr, kw);
    }
    group_sync();
    {
        // every block whose bound is within the tie margin of the best, each block by one warp
        const unsigned kb = S.thr;
        const float gth = kb ? key_score(kb) - cand_delta(key_score(kb)) : -INFINITY;
        for (int qb = gw * 32; qb < P.nblk; qb += kFDThreads) {
            const int q = qb + lane;
            const bool pass = q < P.nblk && block_zmax<SOFTCAP, PENALTY>(__ldcg(bmx + q), P) >= gth;
            unsigned bal = __ballot_sync(0xffffffffu, pass);
            while (bal != 0u) {
                const int qq = qb + __ffs(bal) - 1;
                bal &= bal - 1u;
                scan(qq, gth);
            }
        }
    }
    t = top2_warp_reduce(t);
    if (lane == 0) S.top[gw] = t;
    group_sync();
    if (gt == 0) {
        Top2 tw = S.top[0];
        for (int w = 1; w < kFDWarps; ++w) tw = top2_merge(tw, S.top[w]);
        int y = tw.i1;
        if (tw.i2 >= 0 && tw.s2 >= tw.s1 - cand_delta(tw.s1)) {
            count_diag(P, SPECNG_DIAG_GREEDY_F64);
            const double z1 = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, tw.i1), pen_of(tw.i1), P);
            const double z2 = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, tw.i2), pen_of(tw.i2), P);
            if (better64(z2, tw.i2, z1, tw.i1)) y = tw.i2;
        }
        S.ival[0] = y;
    }
    group_sync();
    return S.ival[0];
}

// Gumbel-max over row a of sequence b (T > 0):
//   DENSE = false: argmax_v (z_v / T - ln E_v) over v != ex (the point-mass
//     residual after rejecting draft ex, or the bonus sample with ex = -1);
//   DENSE = true: argmax_v (log max(0, p_v - q_v) - ln E_v), the residual of a
//     rejected dense draft; returns -2 when the fp32 normaliser cannot settle
//     the decision (the caller then passes the exact one, EXACT = true), -1
//     when the residual is zero everywhere.
// The streaming pass stored every block's bound z_max / T - ln M of its
// scores (log w_v - ln E_v <= z_v / T [- lse] - ln M), so only the blocks
// whose bound reaches the best score found so far are read again.  Seed:
// each warp scores, in its block with the largest bound, each lane's largest
// element; then each warp walks tiles of 32 bounds and reads the passing
// blocks fused_batch at a time (all loads in flight, the block draws made
// meanwhile), screening them against one raw-logit threshold per block
// before the exact per-element score.  Whole group; returns the winner.
template <bool BF16, bool SOFTCAP, bool PENALTY, bool DENSE, bool EXACT = false>
__device__ __noinline__ int group_sample(const VerifyDev& P, DShared& S, const int* pkey, const int* ppos, uint4* stg_all,
                                         int b, int a, int ex, double lse64 = 0.0) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int BLK = 1 << kNoiseBlockShift;
    constexpr int VPL = fused_vpl<BF16>();
    constexpr int NE = VPL * EPV;  // elements per lane per block
    constexpr int NB = fused_batch<BF16>();
    static_assert(NB * NE <= 64, "one 64-bit candidate mask per batch");
    const int gt = threadIdx.x - kFD0 * 32, gw = gt >> 5, lane = gt & 31;
    const int K1 = P.K + 1;
    const size_t row = static_cast<size_t>(b) * K1 + a;
    const float* bnd = P.bmax + row * P.nblk;
    const char* rowp = static_cast<const char*>(P.logits) + row * P.V * ElemTraits<BF16>::SIZE;
    const float* qrow = DENSE ? P.q + (static_cast<size_t>(b) * P.K + a) * P.V : nullptr;
    uint4* stg = stg_all + gw * (NB * 32 * VPL);
    NoiseKey nk = noise_key(P);
    nk.seq = static_cast<uint32_t>(b);
    const RowPhilox rp = row_philox(nk, static_cast<uint32_t>(a));
    auto pen_of = [&](int v) { return PENALTY && pen_lookup(pkey, ppos, S.d, S.nh, P.W, v, a); };
    float lse_f = 0.0f;
    float2 rms = make_float2(0.0f, 0.0f);
    if constexpr (DENSE) {
        rms = __ldcg(reinterpret_cast<const float2*>(&P.rowres[row]));
        lse_f = EXACT ? static_cast<float>(lse64) : rms.x * P.invT + logf(rms.y);
    }
    const float off = DENSE ? lse_f : 0.0f;  // block bounds of the residual: minus lse
    // exact residual score of id v in fp64 (the row's exact normaliser), -inf for a zero residual
    auto exact_residual_score = [&](int v) -> double {
        const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, v), pen_of(v), P);
        const double rsd = exp(z / P.Td - lse64) - static_cast<double>(qrow[v]);
        if (!(rsd > 0.0)) return -INFINITY;
        return log(rsd) - log(noise_exp_f64(nk, static_cast<uint32_t>(v), static_cast<uint32_t>(a)));
    };
    // score of element v (raw logit x) with its own draw, or -inf when it cannot win
    auto score_of = [&](int v, float x, float Mq, int Iq, float thr) -> float {
        const float lnMq = ln_fast(Mq);
        float lw = transform_f32<SOFTCAP, PENALTY>(x, pen_of(v), P) * P.invT;
        if constexpr (DENSE) {
            lw -= lse_f;
            if (lw - lnMq + bound_slack(lw - lnMq) < thr) return -INFINITY;
            if constexpr (EXACT) {
                // in fp64 throughout (the fp32 logarithm of a residual near zero is not
                // accurate enough here); its fp32 rounding only orders the candidates
                return static_cast<float>(exact_residual_score(v));
            }
            lw = log_residual(lw, __ldg(qrow + v));
            if (!(lw > -INFINITY)) return -INFINITY;
        }
        if (lw - lnMq + bound_slack(lw - lnMq) < thr) return -INFINITY;
        return lw - ln_fast(noise_exp_f32(rp, Mq, Iq, static_cast<uint32_t>(v)));
    };
    if (gt == 0) S.thr = 0u;
    group_sync();
    // ---- seed (only sets the threshold; the pass below finds its elements again):
    //      each warp takes up to kSeed blocks with the largest bounds among its lanes'
    //      best ones, and each lane scores its largest element of each (all loads in
    //      flight together, the blocks' draws made meanwhile)
    {
        constexpr int kSeed = 4;
        float lb = -INFINITY;
        int lq = -1;
        for (int q = gw + kFDWarps * lane; q < P.nblk; q += kFDThreads) {
            const float x = __ldcg(bnd + q);
            if (x > lb) { lb = x; lq = q; }
        }
        int qs[kSeed];
#pragma unroll
        for (int h = 0; h < kSeed; ++h) {
            const unsigned kq = warp_best_key(lb);
            const unsigned own = __ballot_sync(0xffffffffu, kq != 0u && lb > -INFINITY && score_key(lb) == kq);
            const int src = own ? __ffs(own) - 1 : -1;
            qs[h] = src >= 0 ? __shfl_sync(0xffffffffu, lq, src) : -1;
            if (lane == src) lb = -INFINITY;  // that lane's block is taken
        }
        uint4 r[kSeed * VPL];
#pragma unroll
        for (int h = 0; h < kSeed; ++h)
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                const int e0 = qs[h] * BLK + (u * 32 + lane) * EPV;
                r[h * VPL + u] = (qs[h] >= 0 && e0 < P.V) ? load_vec_chk<BF16>(P, rowp, e0, P.V)
                                                           : make_uint4(0u, 0u, 0u, 0u);
            }
        int myq = -1;
#pragma unroll
        for (int h = 0; h < kSeed; ++h)
            if (lane == h) myq = qs[h];
        BlockNoise mine{1.0f, 0.0f, 0, 0};
        if (myq >= 0) mine = block_noise(nk, static_cast<uint32_t>(myq), static_cast<uint32_t>(a));
        float sc = -INFINITY;
#pragma unroll
        for (int h = 0; h < kSeed; ++h) {
            const float Mq = __shfl_sync(0xffffffffu, mine.M, h);
            const int Iq = __shfl_sync(0xffffffffu, mine.I, h);
            if (qs[h] < 0) continue;
            float xb = -INFINITY;
            int vb = -1;
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                float x[EPV];
                unpack<BF16>(r[h * VPL + u], x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const int v = qs[h] * BLK + (u * 32 + lane) * EPV + e;
                    if (v < P.V && v != ex && (vb < 0 || x[e] > xb)) { xb = x[e]; vb = v; }
                }
            }
            if (vb >= 0) sc = fmaxf(sc, score_of(vb, xb, Mq, Iq, -INFINITY));
        }
        const unsigned kw = warp_best_key(sc);
        if (kw != 0u && lane == 0) atomicMax(&S.thr, kw);
    }
    group_sync();
    float thr = -INFINITY;
    if (S.thr != 0u) thr = key_score(S.thr) - cand_delta(key_score(S.thr));
    Top2 t = top2_empty();
    // ---- the blocks whose bound reaches the best: a warp's tiles (32 blocks each) are
    //      taken kTG at a time -- all their bounds loaded together and compared with the
    //      threshold (a pass mask per tile) -- then the passing blocks are read again in
    //      batches of NB, across tiles
    constexpr int kTG = 16;
    const int ntiles = P.nblk > gw * 32 ? (P.nblk - gw * 32 + kFDThreads - 1) / kFDThreads : 0;
    for (int tg = 0; tg < ntiles; tg += kTG) {
        {
            float bpf[kTG];
#pragma unroll
            for (int i = 0; i < kTG; ++i) {
                const int q = gw * 32 + (tg + i) * kFDThreads + lane;
                bpf[i] = (tg + i < ntiles && q < P.nblk) ? __ldcg(bnd + q) - off : -INFINITY;
            }
            const unsigned kc = max(*reinterpret_cast<volatile unsigned*>(&S.thr), warp_best_key(t.s1));
            if (kc != 0u) thr = fmaxf(thr, key_score(kc) - cand_delta(key_score(kc)));
#pragma unroll
            for (int i = 0; i < kTG; ++i) {
                const unsigned msk = __ballot_sync(0xffffffffu, bpf[i] > -INFINITY && bpf[i] + bound_slack(bpf[i]) >= thr);
                if (lane == 0) S.pmask[gw][i] = msk;
            }
            __syncwarp();
        }
        int ti = 0;
        unsigned pass = S.pmask[gw][0];
        auto next_block = [&]() -> int {
            while (pass == 0u && ti + 1 < kTG && tg + ti + 1 < ntiles) pass = S.pmask[gw][++ti];
            if (pass == 0u) return -1;
            const int bit = __ffs(pass) - 1;
            pass &= pass - 1u;
            return gw * 32 + (tg + ti) * kFDThreads + bit;
        };
        for (;;) {
            int qh[NB];
#pragma unroll
            for (int h = 0; h < NB; ++h) qh[h] = next_block();
            if (qh[0] < 0) break;
            uint4 r[NB * VPL];
#pragma unroll
            for (int h = 0; h < NB; ++h)
#pragma unroll
                for (int u = 0; u < VPL; ++u) {
                    const int e0 = qh[h] * BLK + (u * 32 + lane) * EPV;
                    r[h * VPL + u] = (qh[h] >= 0 && e0 < P.V) ? load_vec_chk<BF16>(P, rowp, e0, P.V)
                                                               : make_uint4(0u, 0u, 0u, 0u);
                }
            // the batch's block draws, lane h for block h, while the loads are in flight
            int myq = -1;
#pragma unroll
            for (int h = 0; h < NB; ++h)
                if (lane == h) myq = qh[h];
            BlockNoise mine{1.0f, 0.0f, 0, 0};
            if (myq >= 0) mine = block_noise(nk, static_cast<uint32_t>(myq), static_cast<uint32_t>(a));
            float Mh[NB];
            int Ih[NB];
#pragma unroll
            for (int h = 0; h < NB; ++h) {
                Mh[h] = __shfl_sync(0xffffffffu, mine.M, h);
                Ih[h] = __shfl_sync(0xffffffffu, mine.I, h);
            }
            // raw-logit screen per block (none when a penalty below 1 may raise a value)
            float xt[NB];
#pragma unroll
            for (int h = 0; h < NB; ++h)
                xt[h] = qh[h] < 0 ? INFINITY
                                  : ((PENALTY && P.rep < 1.0f) ? -INFINITY
                                                                : raw_screen<SOFTCAP>(thr + off, ln_fast(Mh[h]), P));
#pragma unroll
            for (int i = 0; i < NB * VPL; ++i) stg[i * 32 + lane] = r[i];
            unsigned long long cm = 0ull;
#pragma unroll
            for (int h = 0; h < NB; ++h)
#pragma unroll
                for (int u = 0; u < VPL; ++u) {
                    const uint4 rv = r[h * VPL + u];
                    unsigned bits;
                    if constexpr (BF16) {
                        bits = bf16x8_ge_bits(rv, bf16x2_floor(xt[h]));
                    } else {
                        bits = (__uint_as_float(rv.x) >= xt[h] ? 1u : 0u) | (__uint_as_float(rv.y) >= xt[h] ? 2u : 0u) |
                               (__uint_as_float(rv.z) >= xt[h] ? 4u : 0u) | (__uint_as_float(rv.w) >= xt[h] ? 8u : 0u);
                    }
                    cm |= static_cast<unsigned long long>(bits) << (h * NE + u * EPV);
                }
            __syncwarp();
            while (cm != 0ull) {
                const int bit = __ffsll(static_cast<long long>(cm)) - 1;
                cm &= cm - 1ull;
                const int h = bit / NE, k = bit % NE;
                const int v = qh[h] * BLK + ((k / EPV) * 32 + lane) * EPV + k % EPV;
                if (v >= P.V || v == ex) continue;
                const float xv = elem_of_stage<BF16>(stg, ((h * VPL + k / EPV) * 32 + lane) * EPV + k % EPV);
                const float score = score_of(v, xv, Mh[h], Ih[h], thr);
                if (score > -INFINITY && score >= thr) {  // -inf: a zero weight never wins
                    top2_push(t, score, v);
                    thr = fmaxf(thr, t.s1 - cand_delta(t.s1));
                }
            }
            __syncwarp();
            const unsigned kw = warp_best_key(t.s1);
            if (kw != 0u && lane == 0) atomicMax(&S.thr, kw);
            const unsigned kc = max(*reinterpret_cast<volatile unsigned*>(&S.thr), kw);
            if (kc != 0u) thr = fmaxf(thr, key_score(kc) - cand_delta(key_score(kc)));
        }
    }
    t = top2_warp_reduce(t);
    if (lane == 0) S.top[gw] = t;
    group_sync();
    if (gt == 0) {
        Top2 tw = S.top[0];
        for (int w = 1; w < kFDWarps; ++w) tw = top2_merge(tw, S.top[w]);
        int y = tw.i1;
        const bool close = tw.i2 >= 0 && tw.s2 >= tw.s1 - cand_delta(tw.s1);
        if constexpr (!DENSE) {
            if (close) {
                count_diag(P, SPECNG_DIAG_SAMPLE_F64);
                y = rescore_top2_f64<BF16, SOFTCAP, PENALTY>(P, nk, static_cast<int>(row), a, tw.i1, tw.i2, pen_of(tw.i1),
                                                            pen_of(tw.i2));
            }
        } else if constexpr (EXACT) {
            // every candidate was scored in fp64: only the order of two scores within
            // the fp32 rounding of each other is taken again
            if (close) {
                const double s1 = exact_residual_score(tw.i1), s2 = exact_residual_score(tw.i2);
                y = better64(s2, tw.i2, s1, tw.i1) ? tw.i2 : tw.i1;
            }
        } else if (y >= 0) {
            // fp32 decision when the best is clear of the second and its residual
            // clearly positive (ln p - ln q > 1e-4).  Otherwise the residual's sign or
            // the order of the two may turn on the fp32 normaliser's own error (about
            // 1e-6), which is amplified by 1 / (1 - q / p) near p = q: the caller
            // computes the row's exact normaliser and samples again in fp64 (-2)
            const float x1 = static_cast<float>(raw_logit_chk<BF16>(P, row, tw.i1));
            const float dres = transform_f32<SOFTCAP, PENALTY>(x1, pen_of(tw.i1), P) * P.invT - lse_f - logf(qrow[tw.i1]);
            if (close || !(dres > 1e-4f)) y = -2;
        } else {
            y = -2;  // no positive residual in fp32: confirmed (or not) with the exact normaliser
        }
        S.ival[0] = y;
    }
    group_sync();
    return S.ival[0];
}

// The exact normaliser of row a of sequence b in fp64, the oracle's
// arithmetic: lse = m + ln sum_v exp(z_v / T - m), m = the row's largest
// transformed value / T (from the fp32 record, any reference works).  Whole
// group; a slow full pass over the row, taken only for the rare dense
// residual decisions that the fp32 normaliser cannot settle.
template <bool BF16, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ double group_exact_lse(const VerifyDev& P, DShared& S, const int* pkey, const int* ppos, int b,
                                               int a, double* s_red) {
    const int gt = threadIdx.x - kFD0 * 32, lane = gt & 31, gw = gt >> 5;
    const size_t row = static_cast<size_t>(b) * (P.K + 1) + a;
    const double m = static_cast<double>(__ldcg(&P.rowres[row].m)) / P.Td;
    double acc = 0.0;
    for (int v = gt; v < P.V; v += kFDThreads) {
        const bool pen = PENALTY && pen_lookup(pkey, ppos, S.d, S.nh, P.W, v, a);
        const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, v), pen, P);
        acc += exp(z / P.Td - m);
    }
    acc = warp_sum_f64(acc);
    if (lane == 0) s_red[gw] = acc;
    group_sync();
    double tot = 0.0;
    for (int w = 0; w < kFDWarps; ++w) tot += s_red[w];
    group_sync();
    return m + log(tot);
}

// One completed row (b, j): its test or argmax, the sequence's state, and --
// when this update makes a known -- the token at row a and the outputs.
template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ void group_row_event(const VerifyDev& P, DShared& S, int* pkey, int* ppos, uint4* stg,
                                             const uint8_t* s_keff, int b, int j, int dnext, int pend) {
    const int gt = threadIdx.x - kFD0 * 32, lane = gt & 31;
    const int K1 = P.K + 1;
    const size_t row = static_cast<size_t>(b) * K1 + j;
    const int keff = s_keff[b];
    const bool dense = P.q != nullptr;
    NoiseKey nk = noise_key(P);
    nk.seq = static_cast<uint32_t>(b);
    group_sync();  // every thread has read the arguments the loop passed through S
    // ---- the row's test (T > 0) or argmax (T = 0)
    int acc = 0;
    if constexpr (GREEDY) {
        if (gt < P.K) S.d[gt] = draft_at(P, b, gt);
        group_sync();
        group_load_seq<PENALTY>(P, S, pkey, ppos, b, gt);
        const int y = group_argmax<BF16, SOFTCAP, PENALTY>(P, S, pkey, ppos, b, j);
        if (gt == 0) {
            RowRes rr;
            rr.m = 0.0f; rr.S = 0.0f; rr.winner = y; rr.pad = 0;
            P.rowres[row] = rr;
            const int d = j < keff ? dnext : -1;
            if (j < keff && !(d >= 0 && d < P.V)) raise_status(P.status, SPECNG_DEV_TOKEN_OOR);
            acc = j < keff && d >= 0 && d < P.V && d == y;
        }
    } else if (gt == 0 && j < keff) {
        // the row's normaliser: its one record (reference m, sum relative to it)
        const float2 rec = __ldcg(reinterpret_cast<const float2*>(P.part + row * P.nchunk));
        const float mf = rec.x, Sf = rec.y;
        {
            if (!(Sf > 0.0f && Sf < INFINITY && mf < INFINITY)) raise_status(P.status, SPECNG_DEV_NONFINITE);
            RowRes rr;
            rr.m = mf; rr.S = Sf; rr.winner = -1; rr.pad = 0;
            P.rowres[row] = rr;
            {
                const int d = dnext;
                if (d >= 0 && d < P.V) {
                    const float xd = static_cast<float>(raw_logit_chk<BF16>(P, row, d));
                    const float qdf = dense ? P.q[(static_cast<size_t>(b) * P.K + j) * P.V + chk_id(P, d)] : 1.0f;
                    const double u = accept_uniform_f64(nk, static_cast<uint32_t>(j + 1));
                    const float lsef = mf * P.invT + logf(Sf);
                    const float lp = transform_f32<SOFTCAP, PENALTY>(xd, pend != 0, P) * P.invT - lsef;
                    const float lr = logf(static_cast<float>(u)) + logf(qdf);
                    if (lr < lp - 1e-4f * (1.0f + fabsf(lp))) {
                        acc = 1;
                    } else if (lr > lp + 1e-4f * (1.0f + fabsf(lp))) {
                        acc = 0;
                    } else {
                        count_diag(P, SPECNG_DIAG_ACCEPT_F64);
                        acc = accept_f64<SOFTCAP, PENALTY>(P, xd, pend != 0, u, static_cast<double>(qdf), mf, Sf);
                    }
                } else {
                    raise_status(P.status, SPECNG_DEV_TOKEN_OOR);
                }
            }
        }
    }
    // ---- the sequence's state: this row is done (and accepted)
    if (gt == 0) {
        __threadfence();  // the row record above before the state that announces it
        const unsigned long long bits = (1ull << j) | (acc ? (1ull << (kStateAcc + j)) : 0ull);
        const unsigned long long old = state_or(P.seq_state + b, P.epoch, bits);
        int a = -1;
        if (old == ~0ull) {
            raise_status(P.status, SPECNG_DEV_TIMEOUT);
        } else if (known_a(old, keff) < 0) {
            a = known_a(old | bits, keff);
        }
        __threadfence();  // the other rows' records, announced by their state bits, are read below
        S.ival[1] = a;
    }
    group_sync();
    const int a = S.ival[1];
    if (a < 0) return;
    // ---- the token at row a, then the outputs
    if constexpr (!GREEDY) {
        if (gt < P.K) S.d[gt] = draft_at(P, b, gt);
        group_sync();
        group_load_seq<PENALTY>(P, S, pkey, ppos, b, gt);
    }
    const int da = a < keff ? S.d[a] : -1;
    const bool dvalid = da >= 0 && da < P.V;
    int y;
    if constexpr (GREEDY) {
        y = __ldcg(&P.rowres[static_cast<size_t>(b) * K1 + a].winner);
    } else if (dense && a < keff && dvalid) {
        y = group_sample<BF16, SOFTCAP, PENALTY, true>(P, S, pkey, ppos, stg, b, a, -1);
        if (y == -2) {
            if (gt == 0) count_diag(P, SPECNG_DIAG_RESIDUAL_F64);
            const double lse64 = group_exact_lse<BF16, SOFTCAP, PENALTY>(P, S, pkey, ppos, b, a, S.red);
            y = group_sample<BF16, SOFTCAP, PENALTY, true, true>(P, S, pkey, ppos, stg, b, a, -1, lse64);
        }
        if (y < 0) {
            if (gt == 0) count_diag(P, SPECNG_DIAG_RESIDUAL_ZERO);
            y = group_sample<BF16, SOFTCAP, PENALTY, false>(P, S, pkey, ppos, stg, b, a, -1);
        }
    } else {
        y = group_sample<BF16, SOFTCAP, PENALTY, false>(P, S, pkey, ppos, stg, b, a, (a < keff && dvalid) ? da : -1);
    }
    if (gt < K1) P.out_tokens[static_cast<size_t>(b) * K1 + gt] = gt < a ? S.d[gt] : (gt == a ? y : -1);
    if (gt == 0) {
        int kb = P.k[b];
        if (kb < 0 || kb > P.K) kb = kb < 0 ? 0 : P.K;
        P.out_accept[b] = a;
        P.kv_len[b] = P.kv_len[b] - kb + a;
        float en = __ldcg(P.ema + b);
        if (keff > 0) en = ema_update(en, P.tau, a, keff);
        P.ema_new[b] = en;
        if (P.gate_state != nullptr) P.cool_new[b] = cool_after(P, __ldcg(P.gate_state + b), a, keff);
    }
    group_sync();
}

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kFThreads, 1) verify_fused_kernel(const __grid_constant__ VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = chunk_elems<BF16>();
    constexpr int SB = kChunkBytes;
    constexpr int SL = 32 * kVL * EPV;                          // ids per streaming slice
    constexpr int VPB = (1 << kNoiseBlockShift) / (32 * EPV);   // vector rows per noise block (bf16 1, fp32 2)
    constexpr size_t kPenBytes = PENALTY ? static_cast<size_t>(kStages) * (kChunkBytes / 16) : 0;
    extern __shared__ __align__(128) uint8_t s_dyn[];
    uint8_t* s_stage = s_dyn;
    uint32_t* s_bm = reinterpret_cast<uint32_t*>(s_dyn + kStages * SB);
    uint4* s_stg = reinterpret_cast<uint4*>(s_dyn + kStages * SB + kPenBytes);
    uint16_t* s_ord = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(s_stg) + fused_stage_bytes<BF16>());
    uint8_t* s_keff = reinterpret_cast<uint8_t*>(s_ord + kFusedMaxB);
    int* s_pkey = reinterpret_cast<int*>(s_keff + kFusedMaxB);  // with the penalty: kPenSlots keys, then positions
    int* s_ppos = s_pkey + kPenSlots;
    __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
    __shared__ StageMeta s_meta[kStages];
    __shared__ SegSum s_slot[kStages][kCWarps];
    __shared__ int s_cnt[kStages];
    __shared__ int s_hist[SPECNG_MAX_K + 1];
    __shared__ long long s_off[SPECNG_MAX_K + 2];
    __shared__ int s_hwin[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_pdrafts[SPECNG_MAX_K + 1];
    __shared__ float s_lnm[GREEDY ? 1 : kStages][GREEDY ? 1 : (CHUNK >> kNoiseBlockShift)];
    __shared__ unsigned s_notes[kNoteCap];
    __shared__ int2 s_note_aux[kNoteCap];  // d_{j+1} of the row, and whether it is penalised
    __shared__ unsigned s_note_wr;
    __shared__ int s_stream_done;
    __shared__ int s_last;
    __shared__ DShared S;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    pdl_wait();
    pdl_trigger();

    // ---- prologue: every sequence's k_eff, then the order of the row-chunks
    if (tid <= P.K) s_hist[tid] = 0;
    for (int i = tid; i < kNoteCap; i += kFThreads) s_notes[i] = 0u;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], kCWarps);
            s_cnt[i] = 0;
        }
        mbar_init_fence();
        s_note_wr = 0u;
        s_stream_done = 0;
    }
    __syncthreads();
    for (int b = tid; b < P.B; b += kFThreads) {
        const int ke = gate_keff(P, b, nullptr, blockIdx.x == 0);
        s_keff[b] = static_cast<uint8_t>(ke);
        atomicAdd(&s_hist[ke], 1);
    }
    __syncthreads();
    // stable counting sort by k_eff, largest first: warp v places the sequences with
    // k_eff = v, in increasing b; wave j (rows j of every sequence with k_eff >= j) is
    // then the first W_j entries
    if (warp <= P.K) {
        const int v = warp;
        int pos = 0;
        for (int u = v + 1; u <= P.K; ++u) pos += s_hist[u];
        for (int b0 = 0; b0 < P.B; b0 += 32) {
            const int b = b0 + lane;
            const bool m = b < P.B && s_keff[b] == v;
            const unsigned bal = __ballot_sync(0xffffffffu, m);
            if (m) s_ord[pos + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(b);
            pos += __popc(bal);
        }
    }
    if (tid == 0) {
        // s_off[j]: the first row of wave j in the order (a row is one item)
        long long off = 0;
        int W = 0;
        for (int u = 0; u <= P.K; ++u) W += s_hist[u];
        for (int j = 0; j <= P.K; ++j) {
            s_off[j] = off;
            off += W;
            W -= s_hist[j];
        }
        s_off[P.K + 1] = off;
    }
    __syncthreads();
    const long long N = s_off[P.K + 1];  // rows of the call
    const long long G = gridDim.x;

    if (warp == kPWarp) {
        // ================= producer =================
        constexpr int kHW = PENALTY ? SPECNG_MAX_REP_WINDOW / 32 : 1;
        constexpr int BPC = CHUNK >> kNoiseBlockShift;  // noise blocks per chunk
        constexpr int NPL = GREEDY ? 1 : (BPC + 31) / 32;  // block draws per lane per chunk
        struct Item {
            int b, j, L, draft;
            unsigned long long st;
            int hw[kHW];
            bool valid;
        };
        auto clampL = [&](int L) {
            return L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
        };
        // row t of the order (wave j, rank r): the loads that do not depend on the
        // history length are issued here, two rows before the row is streamed
        auto map_item = [&](long long t, Item& it) {
            it.valid = t < N;
            if (!it.valid) return;
            int j = 0;
            while (j < P.K && t >= s_off[j + 1]) ++j;
            it.j = j;
            it.b = s_ord[t - s_off[j]];
            it.L = PENALTY ? P.lens[it.b] : 0;
            it.draft = lane < P.K ? draft_at(P, it.b, lane) : -1;
            it.st = (P.early_exit && j > 0) ? __ldcg(P.seq_state + it.b) : 0ull;
        };
        // the history tail of the penalty window (first used one row later)
        auto load_tail = [&](Item& it) {
            if constexpr (PENALTY) {
                if (!it.valid) return;
                const int L = clampL(it.L);
                it.L = L;
                const int nh = L < P.W ? L : P.W;
#pragma unroll
                for (int i = 0; i < kHW; ++i) {
                    const int t = lane + 32 * i;
                    it.hw[i] = t < nh ? hist_at(P, it.b, (L - nh) + t) : 0;
                }
            }
        };
        bool ok = true;
        int st = 0, n = 0, issued = 0;
        unsigned eph = 0u;
        // one row into the ring, chunk by chunk (or skipped); false once the ring timed out
        auto issue = [&](const Item& cur) -> bool {
            if (P.early_exit && cur.j > 0) {
                const int a = known_a(state_bits(cur.st, P.epoch), s_keff[cur.b]);
                if (a >= 0 && a < cur.j) return true;  // past a known first rejection
            }
            const int keff = s_keff[cur.b];
            int nh = 0;
            if constexpr (PENALTY) {
                // the window of row j: the history tail, then d_1..d_j
                nh = cur.L < P.W ? cur.L : P.W;
                __syncwarp();  // the previous row's chunks have read the window
#pragma unroll
                for (int i = 0; i < kHW; ++i)
                    if (lane + 32 * i < nh) s_hwin[lane + 32 * i] = cur.hw[i];
                if (lane < keff) s_pdrafts[lane] = cur.draft;
                __syncwarp();
            }
            // the row's draft d_{j+1} (tested when the row is decided) and whether the
            // penalty window of row j holds it
            const int dnext = cur.j < keff ? __shfl_sync(0xffffffffu, cur.draft, cur.j) : -1;
            int pend = 0;
            if constexpr (PENALTY) {
                if (dnext >= 0) {
                    const WindowView wv{s_hwin, s_pdrafts, nh, P.W};
                    pend = wv.warp_has(cur.j, dnext) ? 1 : 0;
                }
            }
            NoiseKey nk = noise_key(P);
            nk.seq = static_cast<uint32_t>(cur.b);
            for (int c = 0; c < P.nchunk; ++c) {
                const int v0 = c * CHUNK;
                const int v1 = min(P.V, v0 + CHUNK);
                const char* src = static_cast<const char*>(P.logits) +
                                  ((static_cast<size_t>(cur.b) * K1 + cur.j) * P.V + v0) * ElemTraits<BF16>::SIZE;
                // the chunk's block draws (ln M of each block minimum), made before the
                // stage is free so that they do not delay it
                float lnm[NPL];
                if constexpr (!GREEDY) {
                    const int blk0 = v0 >> kNoiseBlockShift;
#pragma unroll
                    for (int i = 0; i < NPL; ++i) {
                        const int q = lane + 32 * i;
                        lnm[i] = (q < BPC && blk0 + q < P.nblk)
                                     ? block_noise(nk, static_cast<uint32_t>(blk0 + q), static_cast<uint32_t>(cur.j)).lnM
                                     : 0.0f;
                    }
                }
                if (n >= kStages && !mbar_wait_bounded(&s_empty[st], eph)) {
                    if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT);
                    return false;
                }
                if (P.aligned && lane == 0) {
                    mbar_add_tx(&s_full[st], static_cast<unsigned>(v1 - v0) * ElemTraits<BF16>::SIZE);
                    bulk_g2s(s_stage + st * SB, src, static_cast<unsigned>(v1 - v0) * ElemTraits<BF16>::SIZE, &s_full[st]);
                }
                issued = n + 1;
                StageMeta& mt = s_meta[st];
                if (lane == 0) {
                    mt.b = cur.b; mt.j = cur.j; mt.c = c;
                    mt.seg_end = c == P.nchunk - 1 ? 1 : 0;
                    mt.sum = (!GREEDY && cur.j < keff) ? 1 : 0;
                    mt.dnext = dnext;
                    mt.pend = pend;
                }
                if constexpr (!GREEDY) {
#pragma unroll
                    for (int i = 0; i < NPL; ++i)
                        if (lane + 32 * i < BPC) s_lnm[st][lane + 32 * i] = lnm[i];
                }
                if constexpr (PENALTY) {
                    uint32_t* bm = s_bm + st * (CHUNK / 32);
                    for (int i = lane; i < CHUNK / 32; i += 32) bm[i] = 0u;
                    __syncwarp();
                    const WindowView wv{s_hwin, s_pdrafts, nh, P.W};
                    const int nwin = wv.count(cur.j);
                    unsigned pw = 0u;
                    for (int i = lane; i < nwin; i += 32) {
                        const int tok = wv.token(cur.j, i);
                        if (tok >= v0 && tok < v1) {
                            atomicOr(&bm[(tok - v0) >> 5], 1u << ((tok - v0) & 31));
                            pw |= 1u << ((tok - v0) / SL);
                        }
                    }
                    pw = __reduce_or_sync(0xffffffffu, pw);
                    if (lane == 0) mt.penw = pw;
                } else {
                    if (lane == 0) mt.penw = 0u;
                }
                if (!P.aligned) {
                    uint8_t* dst = s_stage + st * SB;
                    for (int e = lane; e < v1 - v0; e += 32) {
                        if constexpr (BF16) reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(src)[e];
                        else reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(src)[e];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_full[st]);
                ++n;
                if (++st == kStages) {
                    st = 0;
                    if (n > kStages) eph ^= 1u;
                }
            }
            return true;
        };
        // two item slots used in turn (no copies of loads in flight): while one row
        // is issued, the next one's history tail and the one after's lengths load
        long long t = blockIdx.x;
        Item A, Bn;
        map_item(t, A);
        load_tail(A);
        map_item(t + G, Bn);
        while (ok && A.valid) {
            load_tail(Bn);
            ok = issue(A);
            t += G;
            map_item(t + G, A);          // A now holds the row after Bn
            if (!ok || !Bn.valid) break;
            load_tail(A);
            ok = issue(Bn);
            t += G;
            map_item(t + G, Bn);
            if (!ok || !A.valid) break;
        }
        // the end of the stream: a stage whose metadata says so (its item index is n)
        bool marked = false;
        if (ok) {
            if (n >= kStages) ok = mbar_wait_bounded(&s_empty[st], eph);
            if (ok) {
                if (lane == 0) {
                    s_meta[st].b = -1;
                    mbar_arrive(&s_full[st]);
                }
                marked = true;
            } else if (lane == 0) {
                raise_status(P.status, SPECNG_DEV_TIMEOUT);
            }
        }
        // stay until every issued copy has landed: item i completes phase i / kStages of
        // stage i % kStages; the marker's stage already held item n - kStages, which the
        // consumers released, so its copy has landed and that stage is not waited on
        if (P.aligned && lane == 0) {
            int lo = issued > kStages ? issued - kStages : 0;
            if (marked && lo < n - (kStages - 1)) lo = n - (kStages - 1);
            for (int i = lo; i < issued; ++i)
                if (!mbar_wait_bounded(&s_full[i % kStages], static_cast<unsigned>((i / kStages) & 1)))
                    raise_status(P.status, SPECNG_DEV_TIMEOUT);
        }
    } else if (warp < kCWarps) {
        // ================= streaming warps =================
        const int ubase = warp * (32 * kVL);
        const int off0 = ubase * EPV + lane * EPV;
        // the lane's sum of exponentials over the row so far, against a reference m fixed
        // at the row's first value and raised only when a value passes it by more than
        // 2^32 in the sum's units (so the sum never waits for a chunk's maximum)
        float m = -INFINITY, s = 0.0f, msc = 0.0f;
        int st = 0;
        unsigned fph = 0u;
        for (;;) {
            if (!mbar_wait_bounded(&s_full[st], fph)) {
                if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT);
                break;
            }
            const StageMeta& mt = s_meta[st];
            if (mt.b < 0) break;  // end of the stream
            const int c = mt.c;
            const int row = mt.b * K1 + mt.j;
            const bool dosum = !GREEDY && mt.sum != 0;
            const int v0 = c * CHUNK;
            const int v1 = min(P.V, v0 + CHUNK);
            const uint4* stage = reinterpret_cast<const uint4*>(s_stage + st * SB);
            const uint32_t* bm = s_bm + (PENALTY ? st * (CHUNK / 32) : 0);
            const bool full = v0 + off0 + (kVL - 1) * 32 * EPV + EPV <= v1;
            uint4 rv[kVL];
#pragma unroll
            for (int i = 0; i < kVL; ++i) rv[i] = stage[ubase + i * 32 + lane];
            unsigned long long pmk = 0ull;
            if constexpr (PENALTY) {
                if ((mt.penw >> warp) & 1u) {
#pragma unroll
                    for (int i = 0; i < kVL; ++i) {
                        const int off = off0 + i * 32 * EPV;
                        pmk |= static_cast<unsigned long long>((bm[off >> 5] >> (off & 31)) & ((1u << EPV) - 1u)) << (8 * i);
                    }
                }
            }
            uint32_t hv[kVL];
#pragma unroll
            for (int i = 0; i < kVL; ++i) {
                uint4 r = rv[i];
                if (!full) r = mask_tail<BF16>(r, v1 - (v0 + off0 + i * 32 * EPV));
                if constexpr (BF16) {
                    hv[i] = as_u32(bf16x8_max2(r));
                } else {
                    hv[i] = __float_as_uint(fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                                                  fmaxf(__uint_as_float(r.z), __uint_as_float(r.w))));
                }
            }
            if (dosum) {
                if (full) {
                    float lraw;
                    if constexpr (BF16) {
                        uint32_t h = hv[0];
#pragma unroll
                        for (int i = 1; i < kVL; ++i) h = as_u32(__hmax2(as_bf162(h), as_bf162(hv[i])));
                        lraw = fmaxf(bf16lo(h), bf16hi(h));
                    } else {
                        lraw = __uint_as_float(hv[0]);
#pragma unroll
                        for (int i = 1; i < kVL; ++i) lraw = fmaxf(lraw, __uint_as_float(hv[i]));
                    }
                    const float zl = SOFTCAP ? transform_f32<true, false>(lraw, false, P) : lraw;
                    if (!(m > -INFINITY)) {
                        m = zl;
                        msc = m * P.sc;
                    } else if ((zl - m) * P.sc > 32.0f) {
                        // far above the reference: raise it before this chunk's terms
                        s *= ex2_approx((m - zl) * P.sc);
                        m = zl;
                        msc = m * P.sc;
                    }
                    if (m > -INFINITY) {
                        float2 acc2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                                          make_float2(0.0f, 0.0f)};
                        const float2 sc2 = make_float2(P.sc, P.sc), nm2 = make_float2(-msc, -msc);
#pragma unroll
                        for (int i = 0; i < kVL; ++i) {
                            float x[EPV];
                            unpack<BF16>(rv[i], x);
#pragma unroll
                            for (int e = 0; e < EPV; e += 2) {
                                const float2 tt = __ffma2_rn(make_float2(sum_transform<SOFTCAP>(x[e], P),
                                                                         sum_transform<SOFTCAP>(x[e + 1], P)),
                                                             sc2, nm2);
                                acc2[i & 3] = __fadd2_rn(acc2[i & 3], make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
                            }
                        }
                        s += ((acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y)) +
                             ((acc2[2].x + acc2[2].y) + (acc2[3].x + acc2[3].y));
                    }
                    if constexpr (PENALTY) {
                        unsigned long long pw = pmk;
                        while (pw != 0ull) {
                            const int bit = __ffsll(static_cast<long long>(pw)) - 1;
                            pw &= pw - 1ull;
                            const float xe = elem_of_stage<BF16>(stage, off0 + (bit >> 3) * 32 * EPV + (bit & 7));
                            const float zu = sum_transform<SOFTCAP>(xe, P);
                            const float zp = sum_transform_pen<SOFTCAP>(xe, P);
                            if ((zp - m) * P.sc > 32.0f) {
                                s = m > -INFINITY ? s * ex2_approx((m - zp) * P.sc) : 0.0f;
                                m = zp;
                                msc = m * P.sc;
                            }
                            s += ex2_approx(fmaf(zp, P.sc, -msc)) - ex2_approx(fmaf(zu, P.sc, -msc));
                        }
                    }
                } else {
                    const SumState ss = sum_partial<BF16, SOFTCAP, PENALTY>(stage, off0, v0, v1, pmk, SumState{m, s, msc}, P);
                    m = ss.m;
                    s = ss.s;
                    msc = ss.msc;
                }
            }
            // per noise block of my vector rows: at T = 0 its largest raw logit; at T > 0
            // the bound of its sampling scores, z_max / T - ln M (z_max: the transform of
            // the largest raw logit; M: the block's noise minimum, drawn by the producer)
            {
                const int blk0 = (v0 >> kNoiseBlockShift) + warp * (kVL / VPB);
                float* dst = P.bmax + static_cast<size_t>(row) * P.nblk + blk0;
                const int nb = min(kVL / VPB, P.nblk - blk0);
                // lane i < nb finishes block i (all lanes hold the warp-reduced maxima)
                auto bound = [&](float raw) {
                    if constexpr (GREEDY) return raw;
                    return block_zmax<SOFTCAP, PENALTY>(raw, P) * P.invT - s_lnm[st][warp * (kVL / VPB) + lane];
                };
                if constexpr (BF16) {
                    uint32_t bw[kVL / 2];
#pragma unroll
                    for (int p = 0; p < kVL / 2; ++p)
                        bw[p] = as_u32(__hmax2(as_bf162(__byte_perm(hv[2 * p], hv[2 * p + 1], 0x5410)),
                                               as_bf162(__byte_perm(hv[2 * p], hv[2 * p + 1], 0x7632))));
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                        for (int p = 0; p < kVL / 2; ++p)
                            bw[p] = as_u32(__hmax2(as_bf162(bw[p]), as_bf162(__shfl_xor_sync(0xffffffffu, bw[p], off))));
                    float raw = -INFINITY;
#pragma unroll
                    for (int i = 0; i < kVL; ++i)
                        if (lane == i) raw = (i & 1) ? bf16hi(bw[i >> 1]) : bf16lo(bw[i >> 1]);
                    if (lane < nb) dst[lane] = bound(raw);
                } else {
                    float bmv[kVL / VPB];
#pragma unroll
                    for (int p = 0; p < kVL / VPB; ++p) {
                        bmv[p] = __uint_as_float(hv[VPB * p]);
#pragma unroll
                        for (int u = 1; u < VPB; ++u) bmv[p] = fmaxf(bmv[p], __uint_as_float(hv[VPB * p + u]));
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                        for (int p = 0; p < kVL / VPB; ++p) bmv[p] = fmaxf(bmv[p], __shfl_xor_sync(0xffffffffu, bmv[p], off));
                    float raw = -INFINITY;
#pragma unroll
                    for (int p = 0; p < kVL / VPB; ++p)
                        if (lane == p) raw = bmv[p];
                    if (lane < nb) dst[lane] = bound(raw);
                }
            }
            // at the row's last chunk: the warp's (m, s), then the row's record and its
            // hand-over to the decision group by the last warp
            const bool rec = dosum && mt.seg_end;
            if (rec) {
                float pm = m, ps = s;
                if (!(pm > -INFINITY)) ps = 0.0f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float mo = __shfl_xor_sync(0xffffffffu, pm, off);
                    const float so = __shfl_xor_sync(0xffffffffu, ps, off);
                    ms_merge(pm, ps, mo, so, P.sc);
                }
                if (lane == 0) s_slot[st][warp] = SegSum{pm, ps};
            }
            if (mt.seg_end) {
                m = -INFINITY;
                s = 0.0f;
                msc = 0.0f;
            }
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&s_cnt[st], 1) == kCWarps - 1;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                if (rec) {
                    const SegSum wp = lane < kCWarps ? s_slot[st][lane] : SegSum{-INFINITY, 0.0f};
                    float cm = wp.m, cs = wp.s;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float mo = __shfl_xor_sync(0xffffffffu, cm, off);
                        const float so = __shfl_xor_sync(0xffffffffu, cs, off);
                        ms_merge(cm, cs, mo, so, P.sc);
                    }
                    if (lane == 0) P.part[static_cast<size_t>(row) * P.nchunk] = SegSum{cm, cs};  // the row's one record
                }
                if (lane == 0) {
                    s_cnt[st] = 0;
                }
                if (lane == 0 && mt.seg_end) {
                    // the row's last chunk: every warp has finished the row's earlier chunks
                    // (stages are taken in order), so the whole row is streamed; hand it to
                    // the decision group (a slot frees once the group took it)
                    __threadfence_block();
                    const unsigned idx = atomicAdd(&s_note_wr, 1u);
                    volatile unsigned* slot = &s_notes[idx % kNoteCap];
                    bool posted = false;
                    for (int it = 0; it < (1 << 22); ++it) {
                        if (*slot == 0u) {
                            s_note_aux[idx % kNoteCap] = make_int2(mt.dnext, mt.pend);
                            __threadfence_block();
                            *slot = static_cast<unsigned>(row) + 1u;
                            posted = true;
                            break;
                        }
                        if (it >= 32) __nanosleep(64);
                    }
                    if (!posted) raise_status(P.status, SPECNG_DEV_TIMEOUT);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[st]);
            if (++st == kStages) {
                st = 0;
                fph ^= 1u;
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            atomicAdd(&s_stream_done, 1);
        }
    } else {
        // ================= decision group =================
        const int gt = tid - kFD0 * 32;
        unsigned rd = 0u;  // next row (thread 0's copy)
        int idle = 0;
        for (;;) {
            if (gt == 0) {
                int got = -1;
                volatile unsigned* slot = &s_notes[rd % kNoteCap];
                const unsigned v = *slot;
                if (v != 0u) {
                    __threadfence_block();
                    const int2 aux = s_note_aux[rd % kNoteCap];
                    S.ival[3] = aux.x;  // d_{j+1}
                    S.nh = aux.y;       // its penalty flag (S.nh is reloaded before any sampling)
                    *slot = 0u;
                    got = static_cast<int>(v - 1u);
                    ++rd;
                    idle = 0;
                } else {
                    const int sd = *reinterpret_cast<volatile int*>(&s_stream_done);
                    __threadfence_block();  // the count before the slot: a row posted before it is seen
                    if (sd >= kCWarps && *slot == 0u) {
                        got = -2;
                    } else if (++idle > (1 << 22)) {
                        raise_status(P.status, SPECNG_DEV_TIMEOUT);
                        got = -2;
                    } else if (idle > 16) {
                        __nanosleep(128);
                    }
                }
                S.ival[2] = got;
            }
            group_sync();
            const int row = S.ival[2];
            if (row == -2) break;
            if (row >= 0) {
                __threadfence_block();  // the row's records, written by this CTA's streaming warps
                const int dnext = S.ival[3], pend = S.nh;
                group_row_event<BF16, GREEDY, SOFTCAP, PENALTY>(P, S, s_pkey, s_ppos, s_stg, s_keff, row / K1, row % K1,
                                                                dnext, pend);
            }
            group_sync();
        }
    }

    // ---- the grid's last CTA writes the EMAs
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(P.grid_tix, 1u);
        s_last = prev == static_cast<unsigned>(gridDim.x - 1);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int b = tid; b < P.B; b += kFThreads) {
            if (s_keff[b] > 0) P.ema[b] = __ldcg(P.ema_new + b);
            if (P.gate_state != nullptr) P.gate_state[b] = __ldcg(P.cool_new + b);
        }
        if (tid == 0) *P.grid_tix = 0u;
    }
}

}  // namespace specng
