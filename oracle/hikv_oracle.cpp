// ORACLE — test infrastructure only.
//
// A plain, slow, obviously-correct CPU model of the importance-aware,
// budgeted KV-cache decode step.  Only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load it.  It shares no code, header or
// constant with the CUDA library.
//
// Data are fp32 (bf16 inputs widened exactly); every reduction is in double.
// Per unit (layer, batch, KV head) it keeps a list of entries sorted by
// original position; physical order is irrelevant because attention is
// invariant to permuting (k, v) pairs (Kelle summary, sec. 2.2, eq. 1-2).
//
// Step by step, with the passage each follows:
//  * attention      P = softmax(s), s_j = scale * <q_h, k_j>, o_h = sum_j p_hj v_j
//                   (HiKV sec. II-A; Kelle summary sec. 2.2 eq. 1-2).  The scale
//                   is 1/sqrt(d) unless the caller gives one (the pages write
//                   softmax(QK^T) without it; the standard scaled dot product is
//                   the reading taken).
//  * importance     imp_j += sum over the G query heads of the KV group of p_hj
//                   (H2O cumulative score, KV cache compression blog sec. 3
//                   "H2O"; pooled over the query heads sharing a KV head, blog
//                   sec. 5.2; per-head score, Kelle summary sec. 4.1 eq. 3).
//                   The head sum is formed in double and rounded once to
//                   float; the running score is a float32 add.
//  * window score   prefill importance = the attention columns of the last nq
//                   prompt queries, causally masked, summed (HiKV sec. III-D;
//                   SnapKV observation window, blog sec. 3).  Queries are
//                   applied in position order.
//  * recent bank    HiKV Stage I variant of the importance (HiKV sec. III-B,
//                   Algorithm 1 "IS[l] += P_t[l] for l in R"): a decode step
//                   adds attention mass only to tokens of the recent bank --
//                   the W newest positions and the one leaving it this step,
//                   pos >= t - W -- so a token's score is frozen once it is
//                   older.  Eviction is unchanged: of the tokens outside the
//                   window the lowest score goes, ties taking the newest,
//                   which is HiKV's "promote the ejected token only if its
//                   score exceeds the minimum of the important bank".
//  * band score     HiKV's own prefill initialisation (HiKV sec. III-D): each
//                   prompt token's score is its causal attention column
//                   summed over the band of queries from its own position
//                   onward, IS(l) = sum_{k < band} P_{l+k}[l] (the IS
//                   definition of sec. III-B, with band = B_I / 2), queries
//                   past the prompt contributing nothing.
//  * pooled score   SnapKV variant of the prefill score: each token's score
//                   becomes the largest window score of the k_pool positions
//                   starting at its own, S_pooled[i] = max_{0<=m<k} A_obs[i+m]
//                   (blog sec. 3 "SnapKV"), positions with no retained token
//                   (past the end) contributing nothing.
//  * element level  HiKV Stage II (sec. III-C, Algorithm 1), an approximation
//                   switched on by an element budget 0 < B2 < d.  Per query
//                   head, only the B2 dimensions of q with the largest
//                   magnitude (ties: the lower index) enter the logits; the
//                   softmax P of those logits over every retained token feeds
//                   the importance unchanged; for the output, P is cut into
//                   chunks of d consecutive entries in position order, each
//                   chunk keeps its B2 largest entries (ties: the lower
//                   position) and the output is the sum of those p_j v_j, not
//                   renormalised.  A chunk of at most B2 entries keeps all.
//  * eviction       when n > B: sinks (pos < S) and the recent window
//                   (pos > t - W) are always kept; of the rest keep the
//                   B - S - W with the largest importance, ties by lowest
//                   position; the others are evicted (blog sec. 3 "H2O",
//                   StreamingLLM sinks + window; budget per head, HeadKV
//                   summary sec. 3.2).  Survivors keep their scores.
//  * outputs        rounded once from double to the output type (fp32 or bf16
//                   round-to-nearest-even).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Entry {
    int32_t pos;
    float imp;
    std::vector<float> k, v;
};

struct Unit {
    std::vector<Entry> e;            // retained, ascending pos
    std::vector<Entry> last_evicted; // entries removed by the latest evict
    int32_t next_pos = 0;            // positions appended so far
    double evicted_mass = 0.0;       // sum of imp of every evicted entry
};

struct Oracle {
    int L, B, Hq, Hkv, d, G, S, W;
    double scale;
    int out_bf16;
    int nthreads;
    int recent_only = 0;             // HiKV Stage I: accumulate in the recent bank only
    int elem = 0;                    // HiKV Stage II element budget B2 (0: off)
    // [L*B*Hq], latest Stage II decode step: 0 = the chunk selections are
    // certain, 1 = near ties (alts holds every admissible output), 2 = near
    // ties with too many admissible outputs to list
    std::vector<uint8_t> near_tie;
    std::vector<std::vector<float>> alts;   // [L*B*Hq][count * d]
    std::vector<int32_t> budget;     // [L * Hkv]
    std::vector<Unit> units;         // [L][B][Hkv]
    int unit_index(int l, int b, int g) const { return (l * B + b) * Hkv + g; }
    int budget_of(int u) const {
        int g = u % Hkv;
        int l = u / (B * Hkv);
        return budget[l * Hkv + g];
    }
};

// Round a double to the nearest bf16 value (ties to even) and return it as float.
float round_bf16(double x) {
    if (x == 0.0 || !std::isfinite(x)) return (float)x;
    int e;
    double m = std::frexp(x, &e);          // x = m * 2^e, 0.5 <= |m| < 1
    double scaled = m * 256.0;             // 8 significant bits
    double r = std::nearbyint(scaled);     // default mode: ties to even
    return (float)std::ldexp(r / 256.0, e);
}

template <class F>
void parallel_units(int nthreads, int n, F f) {
    if (nthreads <= 1 || n <= 1) {
        for (int i = 0; i < n; ++i) f(i);
        return;
    }
    int t = std::min(nthreads, n);
    std::vector<std::thread> th;
    for (int w = 0; w < t; ++w)
        th.emplace_back([&, w] {
            for (int i = w; i < n; i += t) f(i);
        });
    for (auto& x : th) x.join();
}

// softmax weights of one query over the entries `e` whose pos <= max_pos.
// Returns p (0 for masked entries) and writes the unnormalised output sum.
void attend(const Oracle& O, const std::vector<Entry>& e, const float* q,
            int32_t max_pos, std::vector<double>& p, double* o /* [d] or null */) {
    size_t n = e.size();
    p.assign(n, 0.0);
    std::vector<double> s(n, 0.0);
    double m = -INFINITY;
    for (size_t j = 0; j < n; ++j) {
        if (e[j].pos > max_pos) continue;
        double acc = 0.0;
        for (int c = 0; c < O.d; ++c) acc += (double)q[c] * (double)e[j].k[c];
        s[j] = O.scale * acc;
        m = std::max(m, s[j]);
    }
    double l = 0.0;
    for (size_t j = 0; j < n; ++j)
        if (e[j].pos <= max_pos) l += std::exp(s[j] - m);
    for (size_t j = 0; j < n; ++j)
        if (e[j].pos <= max_pos) p[j] = std::exp(s[j] - m) / l;
    if (o) {
        for (int c = 0; c < O.d; ++c) o[c] = 0.0;
        for (size_t j = 0; j < n; ++j) {
            if (p[j] == 0.0) continue;
            for (int c = 0; c < O.d; ++c) o[c] += p[j] * (double)e[j].v[c];
        }
    }
}

// One chunk of P whose selection a float32 evaluation of the logits could
// decide differently: `sure` entries are kept under every such evaluation,
// `unsure` entries may or may not be, and exactly `pick` of them are.
struct UnsureChunk {
    std::vector<size_t> unsure;
    int pick = 0;
};

// HiKV Stage II attention of one query head over every entry of `e` (which is
// in position order).  Writes the whole softmax P into p and the output of
// the chunk-selected entries into o.
//
// Near ties.  A kernel selects a chunk's largest p by comparing its float32
// logits.  The rounding error of a float32 dot product of the B2 selected
// terms is at most (B2 + 2) * 2^-24 * scale * sum_c |q_c k_jc| (B2 - 1
// additions, the scaling of q, one more for the conversion), doubled here
// for margin.  Where an entry kept by the exact (double) order and one
// dropped by it are closer than their two bounds, either could win in
// float32; every chunk with such pairs is reported in `unsure` (the entries
// in doubt and how many of them are kept), so that a caller can enumerate
// every selection a correct float32 kernel may make.
void attend_stage2(const Oracle& O, const std::vector<Entry>& e, const float* q,
                   std::vector<double>& p, double* o, std::vector<UnsureChunk>* unsure) {
    const int d = O.d, B2 = O.elem;
    const size_t n = e.size();
    // K side: the B2 dimensions of largest |q|, the lower index first on ties
    std::vector<int> dims(d);
    for (int c = 0; c < d; ++c) dims[c] = c;
    std::stable_sort(dims.begin(), dims.end(),
                     [&](int a, int b) { return std::fabs(q[a]) > std::fabs(q[b]); });
    dims.resize(B2);
    std::sort(dims.begin(), dims.end());
    std::vector<double> s(n), err(n);
    double m = -INFINITY;
    const double ulp = std::ldexp(1.0, -24);
    for (size_t j = 0; j < n; ++j) {
        double acc = 0.0, mag = 0.0;
        for (int c : dims) {
            acc += (double)q[c] * (double)e[j].k[c];
            mag += std::fabs((double)q[c] * (double)e[j].k[c]);
        }
        s[j] = O.scale * acc;
        err[j] = 2.0 * (B2 + 2) * ulp * O.scale * mag;
        m = std::max(m, s[j]);
    }
    double l = 0.0;
    for (size_t j = 0; j < n; ++j) l += std::exp(s[j] - m);
    p.assign(n, 0.0);
    for (size_t j = 0; j < n; ++j) p[j] = std::exp(s[j] - m) / l;
    // V side: chunks of d entries, the B2 largest p of each
    std::vector<uint8_t> keep(n, 0);
    for (size_t c0 = 0; c0 < n; c0 += d) {
        const size_t c1 = std::min(n, c0 + (size_t)d);
        if (c1 - c0 <= (size_t)B2) {
            for (size_t j = c0; j < c1; ++j) keep[j] = 1;
            continue;
        }
        std::vector<size_t> idx;
        for (size_t j = c0; j < c1; ++j) idx.push_back(j);
        std::stable_sort(idx.begin(), idx.end(), [&](size_t a, size_t b) { return p[a] > p[b]; });
        for (int r = 0; r < B2; ++r) keep[idx[r]] = 1;
        if (unsure) {
            // lowest a kept entry could read, highest a dropped one could read
            double kept_lo = INFINITY, drop_hi = -INFINITY;
            for (int r = 0; r < B2; ++r) kept_lo = std::min(kept_lo, s[idx[r]] - err[idx[r]]);
            for (size_t r = B2; r < idx.size(); ++r) drop_hi = std::max(drop_hi, s[idx[r]] + err[idx[r]]);
            UnsureChunk uc;
            for (size_t r = 0; r < idx.size(); ++r) {
                const size_t j = idx[r];
                const bool kept = (int)r < B2;
                if (kept ? (s[j] - err[j] <= drop_hi) : (s[j] + err[j] >= kept_lo)) {
                    uc.unsure.push_back(j);
                    if (kept) ++uc.pick;
                }
            }
            if (uc.pick > 0 && uc.unsure.size() > (size_t)uc.pick) unsure->push_back(std::move(uc));
        }
    }
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (size_t j = 0; j < n; ++j) {
        if (!keep[j]) continue;
        for (int c = 0; c < d; ++c) o[c] += p[j] * (double)e[j].v[c];
    }
}

// Every output the selections allowed by `chunks` give: the exact output o
// with, in each unsure chunk, its `pick` kept entries replaced by any `pick`
// of its unsure entries.  Each alternative is rounded to the output type and
// appended to alts ([count][d]).  Returns false when there would be more
// than max_alts alternatives.
bool stage2_alternatives(const Oracle& O, const std::vector<Entry>& e, const std::vector<double>& p,
                         const double* o, const std::vector<UnsureChunk>& chunks, size_t max_alts,
                         std::vector<float>& alts) {
    const int d = O.d;
    // the exact selection's output minus every unsure kept entry
    std::vector<double> base(o, o + d);
    // per chunk: the index sets to try (combinations of `pick` of `unsure`)
    std::vector<std::vector<std::vector<size_t>>> choices;
    size_t total = 1;
    for (const auto& uc : chunks) {
        const std::vector<size_t>& un = uc.unsure;
        // the exact selection keeps the `pick` unsure entries of largest p
        std::vector<size_t> by_p(un);
        std::stable_sort(by_p.begin(), by_p.end(), [&](size_t a, size_t b) { return p[a] > p[b]; });
        for (int r = 0; r < uc.pick; ++r)
            for (int c = 0; c < d; ++c) base[c] -= p[by_p[r]] * (double)e[by_p[r]].v[c];
        std::vector<std::vector<size_t>> combos;
        std::vector<int> sel(uc.pick);
        for (int r = 0; r < uc.pick; ++r) sel[r] = r;
        const int m = (int)un.size();
        while (true) {
            std::vector<size_t> cset;
            for (int r : sel) cset.push_back(un[r]);
            combos.push_back(std::move(cset));
            if (combos.size() > max_alts) return false;
            int r = uc.pick - 1;
            while (r >= 0 && sel[r] == m - uc.pick + r) --r;
            if (r < 0) break;
            ++sel[r];
            for (int t = r + 1; t < uc.pick; ++t) sel[t] = sel[t - 1] + 1;
        }
        total *= combos.size();
        if (total > max_alts) return false;
        choices.push_back(std::move(combos));
    }
    std::vector<size_t> ix(choices.size(), 0);
    std::vector<double> acc(d);
    for (size_t a = 0; a < total; ++a) {
        acc = base;
        for (size_t k = 0; k < choices.size(); ++k)
            for (size_t j : choices[k][ix[k]])
                for (int c = 0; c < d; ++c) acc[c] += p[j] * (double)e[j].v[c];
        for (int c = 0; c < d; ++c) alts.push_back(O.out_bf16 ? round_bf16(acc[c]) : (float)acc[c]);
        for (size_t k = 0; k < choices.size(); ++k) {   // next index of the mixed-radix counter
            if (++ix[k] < choices[k].size()) break;
            ix[k] = 0;
        }
    }
    return true;
}

bool range_ok(const Oracle* O, int layer0, int nl) {
    return O && layer0 >= 0 && nl >= 0 && layer0 + nl <= O->L;
}

}  // namespace

extern "C" {

void* ora_create(int L, int B, int Hq, int Hkv, int d, int S, int W,
                 const int32_t* budgets, double scale, int out_bf16, int nthreads) {
    if (L <= 0 || B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return nullptr;
    Oracle* O = new Oracle();
    O->L = L; O->B = B; O->Hq = Hq; O->Hkv = Hkv; O->d = d; O->G = Hq / Hkv;
    O->S = S; O->W = W;
    O->scale = scale > 0 ? scale : 1.0 / std::sqrt((double)d);
    O->out_bf16 = out_bf16;
    O->nthreads = nthreads > 0 ? nthreads : 1;
    O->budget.assign(budgets, budgets + L * Hkv);
    O->units.resize((size_t)L * B * Hkv);
    O->near_tie.assign((size_t)L * B * Hq, 0);
    O->alts.assign((size_t)L * B * Hq, {});
    return O;
}

void ora_destroy(void* h) { delete (Oracle*)h; }

int ora_num_threads(void* h, int n) {
    Oracle* O = (Oracle*)h;
    if (n > 0) O->nthreads = n;
    return O->nthreads;
}

// k, v: [nl][B][Hkv][ntok][d] fp32.  New entries get imp = 0 and the next
// positions of their unit.
int ora_append(void* h, int layer0, int nl, int ntok, const float* k, const float* v) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer0, nl) || ntok < 0) return 1;
    int per_layer = O->B * O->Hkv;
    parallel_units(O->nthreads, nl * per_layer, [&](int i) {
        int u = layer0 * per_layer + i;
        Unit& U = O->units[u];
        const float* kb = k + (size_t)i * ntok * O->d;
        const float* vb = v + (size_t)i * ntok * O->d;
        for (int t = 0; t < ntok; ++t) {
            Entry en;
            en.pos = U.next_pos++;
            en.imp = 0.0f;
            en.k.assign(kb + (size_t)t * O->d, kb + (size_t)(t + 1) * O->d);
            en.v.assign(vb + (size_t)t * O->d, vb + (size_t)(t + 1) * O->d);
            U.e.push_back(std::move(en));
        }
        U.last_evicted.clear();
    });
    return 0;
}

// Prefill importance: q [nl][B][Hq][nq][d] are the queries of the last nq
// appended positions.  Query i (position t-nq+1+i) sees entries with
// pos <= its own position.  Applied in position order.
int ora_score_window(void* h, int layer0, int nl, int nq, const float* q) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer0, nl) || nq < 0) return 1;
    int per_layer = O->B * O->Hkv;
    parallel_units(O->nthreads, nl * per_layer, [&](int i) {
        int u = layer0 * per_layer + i;
        Unit& U = O->units[u];
        int li = i / per_layer, b = (i / O->Hkv) % O->B, g = i % O->Hkv;
        int32_t t = U.next_pos - 1;
        std::vector<double> p, colsum;
        for (int qi = 0; qi < nq; ++qi) {
            int32_t qpos = t - nq + 1 + qi;
            colsum.assign(U.e.size(), 0.0);
            for (int hh = 0; hh < O->G; ++hh) {
                int head = g * O->G + hh;
                const float* qv = q + ((((size_t)li * O->B + b) * O->Hq + head) * nq + qi) * O->d;
                attend(*O, U.e, qv, qpos, p, nullptr);
                for (size_t j = 0; j < U.e.size(); ++j) colsum[j] += p[j];
            }
            for (size_t j = 0; j < U.e.size(); ++j) {
                float inc = (float)colsum[j];
                U.e[j].imp = U.e[j].imp + inc;
            }
        }
    });
    return 0;
}

// HiKV prefill initialisation (HiKV sec. III-D, with the IS definition of
// sec. III-B): every prompt token l gets IS(l) = sum over the band of queries
// i = l .. l + band - 1 (those that exist, i < n) of P_i[l], P_i being query
// i's causal softmax over the tokens at positions <= i, summed over the G
// query heads of the group.  q [nl][B][Hq][n][d] holds the queries of every
// held position 0..n-1; the unit must hold exactly those positions (a prompt
// not yet cut).  The band sum is formed in double and rounded once; the
// running score is a float32 add.
int ora_score_band(void* h, int layer0, int nl, int band, const float* q) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer0, nl) || band < 1) return 1;
    int per_layer = O->B * O->Hkv;
    const int n = (int)O->units[layer0 * per_layer].e.size();
    for (int i = 0; i < nl * per_layer; ++i) {
        const Unit& U = O->units[layer0 * per_layer + i];
        if ((int)U.e.size() != n || U.next_pos != n) return 2;
        for (int j = 0; j < n; ++j)
            if (U.e[j].pos != j) return 2;
    }
    parallel_units(O->nthreads, nl * per_layer, [&](int i) {
        int u = layer0 * per_layer + i;
        Unit& U = O->units[u];
        int li = i / per_layer, b = (i / O->Hkv) % O->B, g = i % O->Hkv;
        std::vector<double> p, is(n, 0.0);
        for (int qi = 0; qi < n; ++qi) {          // query at position qi
            for (int hh = 0; hh < O->G; ++hh) {
                int head = g * O->G + hh;
                const float* qv = q + ((((size_t)li * O->B + b) * O->Hq + head) * n + qi) * O->d;
                attend(*O, U.e, qv, qi, p, nullptr);
                // tokens l whose band l .. l + band - 1 contains qi
                for (int l = std::max(0, qi - band + 1); l <= qi; ++l) is[l] += p[l];
            }
        }
        for (int l = 0; l < n; ++l) {
            float inc = (float)is[l];
            U.e[l].imp = U.e[l].imp + inc;
        }
    });
    return 0;
}

// SnapKV pooling of the current scores: imp[pos p] <- max of the scores of the
// retained positions in [p, p + kpool).  kpool <= 1 leaves them unchanged.
int ora_pool_importance(void* h, int layer0, int nl, int kpool) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer0, nl) || kpool < 0) return 1;
    if (kpool <= 1) return 0;
    int per_layer = O->B * O->Hkv;
    parallel_units(O->nthreads, nl * per_layer, [&](int i) {
        Unit& U = O->units[layer0 * per_layer + i];
        std::vector<float> raw(U.e.size());
        for (size_t j = 0; j < U.e.size(); ++j) raw[j] = U.e[j].imp;
        for (size_t j = 0; j < U.e.size(); ++j) {
            float best = raw[j];
            // entries are in ascending position: scan forward while in range
            for (size_t m = j + 1; m < U.e.size() && U.e[m].pos < U.e[j].pos + kpool; ++m)
                best = std::max(best, raw[m]);
            U.e[j].imp = best;
        }
    });
    return 0;
}

// One decode step: q [nl][B][Hq][d] -> out [nl][B][Hq][d] (float values,
// rounded to the output type).  Every retained entry is attended,
// including the one appended for this step.
int ora_decode(void* h, int layer0, int nl, const float* q, float* out) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer0, nl)) return 1;
    int per_layer = O->B * O->Hkv;
    for (int i = 0; i < nl * per_layer; ++i)
        if (O->units[layer0 * per_layer + i].e.empty()) return 2;
    parallel_units(O->nthreads, nl * per_layer, [&](int i) {
        int u = layer0 * per_layer + i;
        Unit& U = O->units[u];
        int li = i / per_layer, b = (i / O->Hkv) % O->B, g = i % O->Hkv;
        std::vector<double> p, colsum(U.e.size(), 0.0), o(O->d);
        for (int hh = 0; hh < O->G; ++hh) {
            int head = g * O->G + hh;
            size_t row = (((size_t)li * O->B + b) * O->Hq + head) * O->d;
            if (O->elem > 0 && O->elem < O->d) {
                std::vector<UnsureChunk> unsure;
                attend_stage2(*O, U.e, q + row, p, o.data(), &unsure);
                const size_t hr = (size_t)u / O->Hkv * O->Hq + head;
                O->alts[hr].clear();
                O->near_tie[hr] = 0;
                if (!unsure.empty())
                    O->near_tie[hr] = stage2_alternatives(*O, U.e, p, o.data(), unsure, 4096, O->alts[hr]) ? 1 : 2;
            } else {
                attend(*O, U.e, q + row, INT32_MAX, p, o.data());
            }
            for (size_t j = 0; j < U.e.size(); ++j) colsum[j] += p[j];
            for (int c = 0; c < O->d; ++c)
                out[row + c] = O->out_bf16 ? round_bf16(o[c]) : (float)o[c];
        }
        const int32_t t = U.next_pos - 1;   // this step's token
        for (size_t j = 0; j < U.e.size(); ++j) {
            if (O->recent_only && U.e[j].pos < t - O->W) continue;   // frozen (important bank)
            float inc = (float)colsum[j];
            U.e[j].imp = U.e[j].imp + inc;
        }
    });
    return 0;
}

// Importance rule of decode steps: 0 = H2O cumulative (every retained token),
// 1 = HiKV recent bank only.
int ora_set_recent_only(void* h, int on) {
    Oracle* O = (Oracle*)h;
    O->recent_only = on ? 1 : 0;
    return 0;
}

// HiKV Stage II element budget of decode steps: 0 (or d) = exact attention,
// 0 < b2 < d = the element-level approximation.
int ora_set_element_budget(void* h, int b2) {
    Oracle* O = (Oracle*)h;
    if (!O || b2 < 0 || b2 > O->d) return 1;
    O->elem = b2;
    return 0;
}

// Per query head of layers [layer0, layer0 + nl), for the latest Stage II
// decode step: 0 where every chunk selection is certain under float32
// rounding of the logits, 1 where some is not (ora_stage2_alternatives lists
// the admissible outputs), 2 where there were too many to list.  [nl][B][Hq].
int ora_stage2_near_ties(void* h, int layer0, int nl, uint8_t* flags) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer0, nl)) return 1;
    const size_t per = (size_t)O->B * O->Hq;
    std::memcpy(flags, O->near_tie.data() + (size_t)layer0 * per, (size_t)nl * per);
    return 0;
}

// The admissible outputs of query head `head` of (layer, batch) at the latest
// Stage II decode step, each rounded to the output type: [count][d] into out
// (room for max rows).  Returns count (0 when the selection was certain), or
// -1 when they do not fit or were too many to list.
int ora_stage2_alternatives(void* h, int layer, int b, int head, float* out, int max) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer, 1) || b < 0 || b >= O->B || head < 0 || head >= O->Hq) return -1;
    const size_t hr = ((size_t)layer * O->B + b) * O->Hq + head;
    if (O->near_tie[hr] == 2) return -1;
    const int count = (int)(O->alts[hr].size() / O->d);
    if (count > max) return -1;
    std::memcpy(out, O->alts[hr].data(), O->alts[hr].size() * sizeof(float));
    return count;
}

// Cut every unit of the range with n > B to exactly B entries.
int ora_evict(void* h, int layer0, int nl) {
    Oracle* O = (Oracle*)h;
    if (!range_ok(O, layer0, nl)) return 1;
    int per_layer = O->B * O->Hkv;
    parallel_units(O->nthreads, nl * per_layer, [&](int i) {
        int u = layer0 * per_layer + i;
        Unit& U = O->units[u];
        U.last_evicted.clear();
        int Bu = O->budget_of(u);
        int n = (int)U.e.size();
        if (n <= Bu) return;
        int32_t t = U.next_pos - 1;
        std::vector<Entry> keep, cand;
        for (auto& en : U.e) {
            bool prot = en.pos < O->S || en.pos > t - O->W;
            if (prot) keep.push_back(std::move(en));
            else cand.push_back(std::move(en));
        }
        std::sort(cand.begin(), cand.end(), [](const Entry& a, const Entry& b) {
            if (a.imp != b.imp) return a.imp > b.imp;
            return a.pos < b.pos;
        });
        int kmid = Bu - (int)keep.size();
        if (kmid < 0) kmid = 0;
        if (kmid > (int)cand.size()) kmid = (int)cand.size();
        for (int j = 0; j < (int)cand.size(); ++j) {
            if (j < kmid) keep.push_back(std::move(cand[j]));
            else {
                U.evicted_mass += cand[j].imp;
                U.last_evicted.push_back(std::move(cand[j]));
            }
        }
        std::sort(keep.begin(), keep.end(),
                  [](const Entry& a, const Entry& b) { return a.pos < b.pos; });
        U.e = std::move(keep);
    });
    return 0;
}

int ora_len(void* h, int u) { return (int)((Oracle*)h)->units[u].e.size(); }
int ora_next_pos(void* h, int u) { return ((Oracle*)h)->units[u].next_pos; }
int ora_num_evicted(void* h, int u) { return (int)((Oracle*)h)->units[u].last_evicted.size(); }
double ora_evicted_mass(void* h, int u) { return ((Oracle*)h)->units[u].evicted_mass; }

// Retained entries of unit u in ascending position.  k/v may be null.
int ora_state(void* h, int u, int32_t* pos, float* imp, float* k, float* v) {
    Oracle* O = (Oracle*)h;
    const Unit& U = O->units[u];
    for (size_t j = 0; j < U.e.size(); ++j) {
        if (pos) pos[j] = U.e[j].pos;
        if (imp) imp[j] = U.e[j].imp;
        if (k) std::memcpy(k + j * O->d, U.e[j].k.data(), sizeof(float) * O->d);
        if (v) std::memcpy(v + j * O->d, U.e[j].v.data(), sizeof(float) * O->d);
    }
    return (int)U.e.size();
}

// Entries removed by the latest evict of unit u.
int ora_evicted(void* h, int u, int32_t* pos, float* imp) {
    const Unit& U = ((Oracle*)h)->units[u];
    for (size_t j = 0; j < U.last_evicted.size(); ++j) {
        pos[j] = U.last_evicted[j].pos;
        imp[j] = U.last_evicted[j].imp;
    }
    return (int)U.last_evicted.size();
}

// Make the retained set of unit u equal to `pos` (n entries), which must be a
// subset of retained + last evicted.  Moves entries between the two lists and
// keeps every score; the evicted-mass total follows the move.  Returns 0 on
// success and leaves the unit unchanged on failure.
int ora_resync(void* h, int u, int n, const int32_t* pos) {
    Oracle* O = (Oracle*)h;
    Unit& U = O->units[u];
    std::vector<int32_t> want(pos, pos + n);
    std::sort(want.begin(), want.end());
    if (std::adjacent_find(want.begin(), want.end()) != want.end()) return 1;
    int found = 0;
    for (auto* list : {&U.e, &U.last_evicted})
        for (auto& en : *list)
            found += std::binary_search(want.begin(), want.end(), en.pos) ? 1 : 0;
    if (found != n) return 1;
    double old_mass = 0.0;
    for (auto& en : U.last_evicted) old_mass += en.imp;
    std::vector<Entry> keep, out;
    for (auto* list : {&U.e, &U.last_evicted})
        for (auto& en : *list) {
            if (std::binary_search(want.begin(), want.end(), en.pos)) keep.push_back(std::move(en));
            else out.push_back(std::move(en));
        }
    std::sort(keep.begin(), keep.end(),
              [](const Entry& a, const Entry& b) { return a.pos < b.pos; });
    double new_mass = 0.0;
    for (auto& en : out) new_mass += en.imp;
    U.evicted_mass += new_mass - old_mass;
    U.e = std::move(keep);
    U.last_evicted = std::move(out);
    return 0;
}

}  // extern "C"
