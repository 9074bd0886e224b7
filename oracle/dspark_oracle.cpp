// dspark_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU restatement of one DSpark decode cycle,
// written in double precision so that a reader can check it against the
// pages by eye.  It exists to produce expected values for the tests, for
// __graft_entry__.smoke() and for the CPU baseline leg of bench.py; the
// product path (the CUDA library) never links, loads or calls it, and this
// file shares no code, header, table or constant generator with it.
//
// Sources (cited by page title and section):
//   [EXPL]  "DSpark: making speculative decoding solve suffix quality and
//           production verify waste" (papers.franksyz.com mainline topic 31),
//           numbered sections 2-10.
//   [PR]    "spec: add DSpark speculative decoding" (llama.cpp pull request
//           25173), description bullets on the draft-dspark type and the
//           Markov head, and the "Losslessness" paragraph.
//   [SC11]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
//           1, 2, 3", SC'11 -- definition of Philox4x32-10.
//
// Readings the pages leave open are the plain ones and are listed in the
// repository's design notes; each is restated where it is used below.
//
// Parity status: every function here is pinned by a CPU test against
// something other than itself (closed forms, brute force, an independent
// library Philox, empirical laws); none is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <limits>

namespace {

// ------------------------------------------------------------------------
// Philox4x32-10 [SC11 section 3]: a 10-round counter-based generator over a
// 128-bit counter (4 x 32-bit words) and a 64-bit key (2 x 32-bit words).
// Each round multiplies counter words 0 and 2 by two fixed odd constants,
// keeps the high and low halves of the 64-bit products, and mixes the high
// halves with the other two counter words and the round key.  The key is
// bumped by two Weyl constants between rounds.
// ------------------------------------------------------------------------
const uint32_t kPhiloxM0 = 0xD2511F53u;
const uint32_t kPhiloxM1 = 0xCD9E8D57u;
const uint32_t kPhiloxW0 = 0x9E3779B9u;
const uint32_t kPhiloxW1 = 0xBB67AE85u;

void philox4x32_10(const uint32_t ctr_in[4], uint32_t key0, uint32_t key1,
                   uint32_t out[4]) {
    uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint32_t k0 = key0, k1 = key1;
    for (int round = 0; round < 10; ++round) {
        const uint64_t prod0 = (uint64_t)kPhiloxM0 * (uint64_t)x0;
        const uint64_t prod1 = (uint64_t)kPhiloxM1 * (uint64_t)x2;
        const uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        const uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        const uint32_t y0 = hi1 ^ x1 ^ k0;
        const uint32_t y1 = lo1;
        const uint32_t y2 = hi0 ^ x3 ^ k1;
        const uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

// The purposes the cycle draws random numbers for.  The counter layout is
// this library's choice (the pages fix none): word 0 = vocabulary index / 4
// (0 for a single draw), word 1 = block position, word 2 = request index,
// word 3 = (cycle << 4) | purpose; key = the request's 64-bit seed.  Because
// every draw is addressed by its own counter, a rejection on one branch never
// shifts the numbers another branch sees (the "RNG desync after different
// rejection branches" failure listed in [EXPL] section 15).
enum Purpose { kDraftGumbel = 0, kAccept = 1, kResidualGumbel = 2, kBonusGumbel = 3 };

// The uniform in (0,1) made from one 32-bit word: the top 23 bits plus one
// half, times 2^-23.  Exact in both float and double.
double uniform_from_bits(uint32_t x) {
    return ((double)(x >> 9) + 0.5) * (1.0 / 8388608.0);
}

uint32_t philox_word(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2,
                     uint32_t c3, int lane) {
    const uint32_t ctr[4] = {c0, c1, c2, c3};
    uint32_t out[4];
    philox4x32_10(ctr, (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32), out);
    return out[lane];
}

// u for vocabulary entry v at (request, position, purpose).
double uniform_vocab(uint64_t seed, uint32_t cycle, int purpose, int req,
                     int pos, int v) {
    const uint32_t w = philox_word(seed, (uint32_t)v >> 2, (uint32_t)pos,
                                   (uint32_t)req, (cycle << 4) | (uint32_t)purpose,
                                   v & 3);
    return uniform_from_bits(w);
}

// u for a single per-position draw (the acceptance test).
double uniform_single(uint64_t seed, uint32_t cycle, int purpose, int req, int pos) {
    const uint32_t w = philox_word(seed, 0u, (uint32_t)pos, (uint32_t)req,
                                   (cycle << 4) | (uint32_t)purpose, 0);
    return uniform_from_bits(w);
}

// Standard Gumbel noise from a uniform: g = -log(-log u).
double gumbel(double u) { return -std::log(-std::log(u)); }

// The draft draw's two uniforms of vocabulary segment s (16 consecutive
// entries, s = v / 16).  The segment is slot j = s % 8 of the 128-entry block
// b = s / 8; slots j and j + 4 share the Philox counter (4 b + j % 4, position,
// request, (cycle << 4) | purpose) and take words (0, 1) when j < 4, (2, 3)
// otherwise: the first word is the race uniform u, the second the in-segment
// uniform a.  (This library's layout; the pages fix none.)
void segment_uniforms(uint64_t seed, uint32_t cycle, int purpose, int req, int pos,
                      int seg, double* u, double* a) {
    const uint32_t blk = (uint32_t)seg >> 3, slot = (uint32_t)seg & 7u;
    const uint32_t ctr[4] = {4u * blk + (slot & 3u), (uint32_t)pos, (uint32_t)req,
                             (cycle << 4) | (uint32_t)purpose};
    uint32_t out[4];
    philox4x32_10(ctr, (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32), out);
    const int w = (slot < 4u) ? 0 : 2;
    *u = uniform_from_bits(out[w]);
    *a = uniform_from_bits(out[w + 1]);
}

double bf16_to_double(uint16_t b) {
    const uint32_t bits = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return (double)f;
}

// Element read for the two storage types the library accepts: 0 = fp32,
// 1 = bf16 (raw 16-bit patterns); 2 = double, for base logits that the
// oracle forms itself (orc_fused_draft).
double load_elem(const void* base, int dtype, size_t idx) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    if (dtype == 2) return ((const double*)base)[idx];
    return bf16_to_double(((const uint16_t*)base)[idx]);
}

// log(sum(exp(x))) with the maximum factored out.
double logsumexp(const double* x, int n) {
    double m = -std::numeric_limits<double>::infinity();
    for (int i = 0; i < n; ++i) m = std::max(m, x[i]);
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += std::exp(x[i] - m);
    return m + std::log(s);
}

// Index of the largest entry (lowest index on ties) and the gap to the
// runner-up; the gap is what decides whether a GPU disagreement is a
// rounding-level near tie.
int argmax_with_gap(const double* x, int n, double* gap) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (x[i] > x[best]) best = i;
    double second = -std::numeric_limits<double>::infinity();
    for (int i = 0; i < n; ++i)
        if (i != best) second = std::max(second, x[i]);
    if (gap) *gap = x[best] - second;
    return best;
}

}  // namespace

extern "C" {

// Status codes shared in meaning (not in code) with the library.
static const int ORC_OK = 0;
static const int ORC_INVALID = -1;
static const int ORC_CAPACITY = -3;
static const int ORC_DEVICE_INPUT = -6;

void orc_philox4x32_10(const uint32_t ctr[4], uint64_t seed, uint32_t out[4]) {
    philox4x32_10(ctr, (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32), out);
}

void orc_philox4x32_10_batch(const uint32_t* ctr, const uint64_t* keys, int n, uint32_t* out) {
    for (int i = 0; i < n; ++i)
        philox4x32_10(ctr + 4 * (size_t)i, (uint32_t)(keys[i] & 0xFFFFFFFFu),
                      (uint32_t)(keys[i] >> 32), out + 4 * (size_t)i);
}

double orc_uniform_from_bits(uint32_t x) { return uniform_from_bits(x); }

double orc_uniform_vocab(uint64_t seed, uint32_t cycle, int purpose, int req,
                         int pos, int v) {
    return uniform_vocab(seed, cycle, purpose, req, pos, v);
}

double orc_uniform_single(uint64_t seed, uint32_t cycle, int purpose, int req, int pos) {
    return uniform_single(seed, cycle, purpose, req, pos);
}

// Markov-head bias for one previous token ([PR] description, draft-dspark
// bullet: bias(prev) = markov_w2 . markov_w1[prev]; with both factors stored
// as [V, rank] rows, b[v] = <W2[v,:], W1[prev,:]>).  Accumulated in double in
// rank order.  prev < 0 means "no previous token": b = 0.
void orc_markov_bias(const void* W1, const void* W2, int w_dtype, int V, int rank,
                     int prev, double* b) {
    for (int v = 0; v < V; ++v) {
        double acc = 0.0;
        if (prev >= 0) {
            for (int j = 0; j < rank; ++j)
                acc += load_elem(W2, w_dtype, (size_t)v * rank + j) *
                       load_elem(W1, w_dtype, (size_t)prev * rank + j);
        }
        b[v] = acc;
    }
}

double orc_logsumexp(const double* x, int n) { return logsumexp(x, n); }

void orc_softmax(const double* x, int n, double* out) {
    const double lse = logsumexp(x, n);
    for (int i = 0; i < n; ++i) out[i] = std::exp(x[i] - lse);
}

// The residual weights used after a rejection ([EXPL] section 3: keep only
// the mass the target has beyond the drafter, max(0, p - q); sampling from
// the full p would count the overlap twice).  Returns their sum.
double orc_residual_weights(const double* p, const double* q, int n, double* res) {
    double total = 0.0;
    for (int i = 0; i < n; ++i) {
        res[i] = std::max(0.0, p[i] - q[i]);
        total += res[i];
    }
    return total;
}

// One semi-autoregressive Markov-head block draft for R requests
// ([EXPL] sections 6-7: drafter logits are the backbone's base logits U_k plus
// a bias B_k that depends on the in-block prefix; the Markov head looks at the
// previous sampled token only.  [PR] description: the block is anchor-first
// -- position 0 already predicts the first draft token -- and is sampled left
// to right with bias(prev)).
//
// For k = 0..gamma-1 and every request r:
//   prev   = anchor[r] at k = 0, else y[r][k-1]   (anchor < 0: no bias at k=0)
//   s_v    = (U[r][k][v] + b_v(prev)) * invT      (T > 0)
//          =  U[r][k][v] + b_v(prev)              (T = 0, greedy)
//   y      = argmax_v s_v (lowest index on ties)                         (T = 0)
//          = a draw from q = softmax(s) by Gumbel-max                    (T > 0)
//   q_lse  = logsumexp_v s_v ;  q_tok = exp(s_y - q_lse)
//
// The Gumbel-max draw builds its noise top-down (Maddison, Tarlow, Minka,
// "A* Sampling", NIPS 2014, section 3: for any partition of the entries, the
// largest perturbed logit of a part is a Gumbel variable located at the log of
// the part's total weight, and which entry attains it is independent of that
// value and has probability w_v / W_part).  With parts = segments of 16
// consecutive entries (the last one ragged) and (u_s, a_s) the segment's two
// uniforms (segment_uniforms, purpose 0, position k):
//   W_s    = sum_{v in s} exp(s_v)
//   race   = log W_s - log(-log u_s)  ->  s* = argmax (lowest segment on ties)
//   y      = the first v in s* whose running sum of exp(s_v') over s* up to
//            and including v exceeds a_{s*} W_{s*}
// so y is the argmax of a Gumbel-perturbed q, like one uniform per entry,
// with two uniforms per 16 entries.
// invT is the fp32 value 1.0f/T, shared with the library, widened to double.
// req_ids maps the rows given here to the request indices the random
// counters use (NULL: identity), so a subset of a batch can be replayed.
// margin[r][k] receives how close the decision came to another token: greedy,
// the gap between the two largest logits; sampling, the smaller of the gap
// between the two best segment race values and the distance of a W from the
// running sums on either side of y, in units of W.
int orc_markov_draft(const void* U, int u_dtype, const void* W1, const void* W2,
                     int w_dtype, const int32_t* anchor, const uint64_t* seeds,
                     const int32_t* req_ids, uint32_t cycle, float temperature,
                     int R, int gamma, int V, int rank,
                     int32_t* y, double* q_lse, double* q_tok,
                     double* q_logits, double* margin) {
    if (R <= 0 || gamma <= 0 || V <= 0 || rank <= 0 || !(temperature >= 0.0f))
        return ORC_INVALID;
    const bool greedy = temperature == 0.0f;
    const double invT = greedy ? 1.0 : (double)(1.0f / temperature);
    std::vector<double> b(V), s(V);
    for (int r = 0; r < R; ++r) {
        const int rid = req_ids ? req_ids[r] : r;
        for (int k = 0; k < gamma; ++k) {
            const int prev = (k == 0) ? anchor[r] : y[(size_t)r * gamma + k - 1];
            if (prev >= V) return ORC_DEVICE_INPUT;
            orc_markov_bias(W1, W2, w_dtype, V, rank, prev, b.data());
            for (int v = 0; v < V; ++v) {
                const double base = load_elem(U, u_dtype, ((size_t)r * gamma + k) * V + v);
                s[v] = greedy ? (base + b[v]) : (base + b[v]) * invT;
            }
            double gap = 0.0;
            int tok = 0;
            const double lse = logsumexp(s.data(), V);
            if (greedy) {
                tok = argmax_with_gap(s.data(), V, &gap);
            } else {
                // the segments' race values (weights relative to exp(lse))
                const int n_seg = (V + 15) / 16;
                std::vector<double> race(n_seg), a_of(n_seg), W(n_seg);
                for (int g = 0; g < n_seg; ++g) {
                    double u, a;
                    segment_uniforms(seeds[r], cycle, kDraftGumbel, rid, k, g, &u, &a);
                    double w_sum = 0.0;
                    for (int v = 16 * g; v < std::min(V, 16 * g + 16); ++v) w_sum += std::exp(s[v] - lse);
                    W[g] = w_sum;
                    a_of[g] = a;
                    race[g] = w_sum > 0.0 ? std::log(w_sum) - std::log(-std::log(u))
                                          : -std::numeric_limits<double>::infinity();
                }
                const int win = argmax_with_gap(race.data(), n_seg, &gap);
                if (n_seg == 1) gap = std::numeric_limits<double>::infinity();
                // the entry of the winning segment by its running sum
                const double target = a_of[win] * W[win];
                double run = 0.0, before = 0.0;
                tok = std::min(V, 16 * win + 16) - 1;
                for (int v = 16 * win; v < std::min(V, 16 * win + 16); ++v) {
                    before = run;
                    run += std::exp(s[v] - lse);
                    if (run > target) { tok = v; break; }
                }
                gap = std::min(gap, std::min(target - before, run - target) / W[win]);
            }
            y[(size_t)r * gamma + k] = tok;
            if (q_lse) q_lse[(size_t)r * gamma + k] = lse;
            if (q_tok) q_tok[(size_t)r * gamma + k] = std::exp(s[tok] - lse);
            if (margin) margin[(size_t)r * gamma + k] = gap;
            if (q_logits)
                std::memcpy(q_logits + ((size_t)r * gamma + k) * V, s.data(), sizeof(double) * V);
        }
    }
    return ORC_OK;
}

// Block draft from the drafter's hidden states, with the base logits formed
// here instead of given ([EXPL] section 6: the parallel backbone produces
// every block position's hidden state in one pass, and the base logits U_k
// come from it; [PR] description: the drafter shares the target's lm_head).
// Written out:
//   U[r][k][v] = sum_i W_lm[v][i] * h[r][k][i]     (double, i = 0 .. d-1 in order)
// and then every step of orc_markov_draft on those base logits, so that
//   s_v = (U[r][k][v] + sum_j W2[v][j] * W1[prev][j]) * invT
// is one contraction over the concatenated K = d + rank.
//   h     [R, gamma, d]   x_dtype (0 fp32, 1 bf16): hidden state of request r at
//                         block position k (rows of the requests given, like U)
//   W_lm  [V, d]          x_dtype: the shared lm_head, one row per vocabulary entry
// Everything else, outputs included, as orc_markov_draft.
int orc_fused_draft(const void* h, const void* W_lm, int x_dtype, int d, const void* W1,
                    const void* W2, int w_dtype, const int32_t* anchor, const uint64_t* seeds,
                    const int32_t* req_ids, uint32_t cycle, float temperature,
                    int R, int gamma, int V, int rank,
                    int32_t* y, double* q_lse, double* q_tok, double* q_logits, double* margin) {
    if (R <= 0 || gamma <= 0 || V <= 0 || d <= 0 || rank <= 0) return ORC_INVALID;
    std::vector<double> U((size_t)R * gamma * V);
    for (int r = 0; r < R; ++r)
        for (int k = 0; k < gamma; ++k) {
            const size_t hrow = ((size_t)r * gamma + k) * d;
            for (int v = 0; v < V; ++v) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i)
                    acc += load_elem(W_lm, x_dtype, (size_t)v * d + i) * load_elem(h, x_dtype, hrow + i);
                U[((size_t)r * gamma + k) * V + v] = acc;
            }
        }
    return orc_markov_draft(U.data(), 2, W1, W2, w_dtype, anchor, seeds, req_ids, cycle, temperature,
                            R, gamma, V, rank, y, q_lse, q_tok, q_logits, margin);
}

// Lossless verification of R drafted blocks ([EXPL] section 2: verify left
// to right, discard everything after the first rejection, emit a correction
// from the residual on rejection or a bonus token from the target's next
// distribution when every draft is accepted; section 3: accept draft v with
// probability min(1, p(v)/q(v)), residual max(0, p - q) renormalised;
// section 13: the verified rows of all requests are packed back to back with
// boundary markers instead of padding).
//
// Target rows of request r are cu_seqlens[r] .. cu_seqlens[r+1]-1; there are
// l_r + 1 of them, l_r in [0, gamma] drafts to verify plus the row after them.
//   t      = target_row * invT          (T > 0; at T = 0 the row itself)
//   p      = softmax(t) ;  q = softmax(q_logits[r][j]) (the drafter's scaled logits)
//   accept draft j iff u_j < p(y_j) / q(y_j), u_j = Philox(purpose 1, position j)
//   greedy: accept iff y_j == argmax(target row j)
// First rejection at j: token ~ max(0, p - q) by Gumbel-max on log weights
// (purpose 2, position j); if that residual is empty in double the token is
// drawn from p with the same noise (counted in residual_empty).  Every draft
// accepted: bonus token ~ p of row l_r (purpose 3, position l_r).  Greedy:
// the argmax of row n_acc.
// out_tokens[r] = y[r][0 .. n_acc-1], token, then -1 up to gamma+1 entries.
// accept_margin[r][j] = |u_j - ratio| (greedy: the target row's top-two gap);
// sample_margin[r]    = top-two gap of the scores that chose the last token.
int orc_verify(const float* target, const int32_t* cu_seqlens, const int32_t* y,
               const double* q_logits, const uint64_t* seeds, const int32_t* req_ids,
               uint32_t cycle, float temperature, int R, int gamma, int V,
               int32_t* n_acc, int32_t* out_tokens, double* p_tok,
               double* accept_margin, double* sample_margin, int32_t* residual_empty) {
    if (R <= 0 || gamma <= 0 || V <= 0 || !(temperature >= 0.0f)) return ORC_INVALID;
    const bool greedy = temperature == 0.0f;
    const double invT = greedy ? 1.0 : (double)(1.0f / temperature);
    std::vector<double> t(V), p(V), q(V), res(V), score(V);
    int status = ORC_OK;
    for (int r = 0; r < R; ++r) {
        const int rid = req_ids ? req_ids[r] : r;
        const int l = cu_seqlens[r + 1] - cu_seqlens[r] - 1;
        int32_t* out = out_tokens + (size_t)r * (gamma + 1);
        for (int j = 0; j <= gamma; ++j) out[j] = -1;
        if (residual_empty) residual_empty[r] = 0;
        if (l < 0 || l > gamma) { n_acc[r] = -1; status = ORC_DEVICE_INPUT; continue; }
        bool bad = false;
        for (int j = 0; j < l; ++j) {
            const int yj = y[(size_t)r * gamma + j];
            if (yj < 0 || yj >= V) bad = true;
        }
        if (bad) { n_acc[r] = -1; status = ORC_DEVICE_INPUT; continue; }

        auto load_row = [&](int j) {
            const float* row = target + (size_t)(cu_seqlens[r] + j) * V;
            for (int v = 0; v < V; ++v) t[v] = greedy ? (double)row[v] : (double)row[v] * invT;
        };

        int n = l;
        for (int j = 0; j < l; ++j) {
            const int yj = y[(size_t)r * gamma + j];
            load_row(j);
            double gap = 0.0;
            const int amax = argmax_with_gap(t.data(), V, &gap);
            bool accept;
            if (greedy) {
                if (p_tok) p_tok[(size_t)r * gamma + j] = (yj == amax) ? 1.0 : 0.0;
                accept = (yj == amax);
                if (accept_margin) accept_margin[(size_t)r * gamma + j] = gap;
            } else {
                const double lse_p = logsumexp(t.data(), V);
                const double pt = std::exp(t[yj] - lse_p);
                const double* ql = q_logits + ((size_t)r * gamma + j) * V;
                const double lse_q = logsumexp(ql, V);
                const double qt = std::exp(ql[yj] - lse_q);
                const double ratio = pt / qt;
                const double u = uniform_single(seeds[r], cycle, kAccept, rid, j);
                if (p_tok) p_tok[(size_t)r * gamma + j] = pt;
                if (accept_margin) accept_margin[(size_t)r * gamma + j] = std::fabs(u - ratio);
                accept = u < ratio;
            }
            if (!accept) { n = j; break; }
        }
        for (int j = n + 1; j < l && accept_margin; ++j)
            accept_margin[(size_t)r * gamma + j] = std::numeric_limits<double>::infinity();
        n_acc[r] = n;
        for (int j = 0; j < n; ++j) out[j] = y[(size_t)r * gamma + j];

        load_row(n);
        double gap = 0.0;
        int tok;
        if (greedy) {
            tok = argmax_with_gap(t.data(), V, &gap);
        } else if (n < l) {
            orc_softmax(t.data(), V, p.data());
            orc_softmax(q_logits + ((size_t)r * gamma + n) * V, V, q.data());
            const double mass = orc_residual_weights(p.data(), q.data(), V, res.data());
            const bool empty = !(mass > 0.0);
            if (empty && residual_empty) residual_empty[r] = 1;
            for (int v = 0; v < V; ++v) {
                const double g = gumbel(uniform_vocab(seeds[r], cycle, kResidualGumbel, rid, n, v));
                if (empty)
                    score[v] = t[v] + g;
                else
                    score[v] = (res[v] > 0.0) ? std::log(res[v]) + g
                                              : -std::numeric_limits<double>::infinity();
            }
            tok = argmax_with_gap(score.data(), V, &gap);
        } else {
            for (int v = 0; v < V; ++v)
                score[v] = t[v] + gumbel(uniform_vocab(seeds[r], cycle, kBonusGumbel, rid, l, v));
            tok = argmax_with_gap(score.data(), V, &gap);
        }
        out[n] = tok;
        if (sample_margin) sample_margin[r] = gap;
    }
    return status;
}

// Survival, capacity and prefix-closed selection ([EXPL] section 5: the value
// of a suffix position is the product of the conditional acceptance rates;
// section 8: a[r,k] = cumulative product of c[r,k]; section 9: choose
// prefix-closed verify lengths l[r] maximising predicted output times the
// engine's step rate SPS(B), B = physical query rows; the theoretical greedy
// adds candidates in order of a and stops when Theta stops improving;
// section 10: the production design fixes the physical capacity K from the
// confidences of two steps earlier and takes the top-K prefixes of the
// current a within it).
//
//   a[r][k]   = a[r][k-1] * c[r][k] (fp32, a[r][0] = c[r][0])
//   order     = a descending, then k ascending, then r ascending
//   Theta(n)  = SPS(Bpad) * (R + sum of the n best a), Bpad = smallest capture
//               size >= R + n (the R term is the one target-correct token
//               every request gets, section 2)
//   mode 0 (fixed)     : n = min(K_cap - R, R*gamma)
//   mode 1 (history)   : for every capture size S >= R, n_S = min(min(S,K_cap) - R, R*gamma);
//                        pick S maximising SPS_S * (R + sum of the n_S best a_hist)
//                        (ties: the smaller S); n = n_S
//   mode 2 (current)   : as mode 1 on the current a (anticipating; kept for study)
//   mode 3 (first stop): from n = 0, add the next candidate while Theta strictly
//                        grows, B <= K_cap and a capture size >= B exists
//   mode 4 (confidence cutoff): the static per-request cutoff of the llama.cpp
//                        PR's confidence pruning (conf_min) and of the Strata
//                        plan's first scheduling milestone: request r is
//                        eligible up to its first position with c[r][k] < conf_min
//   mode 5 (survival cutoff): eligible where a[r][k] >= conf_min (a fixed
//                        per-request threshold on the survival, the baseline
//                        [EXPL] section 9 compares the global scheduler with)
//                        modes 4 and 5: n = min(eligible, K_cap - R), the n best
//                        eligible candidates in the same order
// The n best current candidates are selected; l[r] counts them per request;
// cu_seqlens[r+1] = cu_seqlens[r] + l[r] + 1; K_used = R + n.
// theta_gap receives the relative gap between the best and second-best Theta
// of the capacity choice (modes 1-3; +inf when there is no alternative).
int orc_select_prefix(const float* c, const float* c_hist, const int32_t* capture_sizes,
                      const float* sps, int n_steps, int K_cap, int mode, float conf_min, int R,
                      int gamma, float* a, int32_t* l, int32_t* cu_seqlens, int32_t* K_used,
                      double* theta_gap) {
    if (R <= 0 || gamma <= 0 || !c || mode < 0 || mode > 5) return ORC_INVALID;
    if (mode == 1 && !c_hist) return ORC_INVALID;
    if (mode >= 1 && mode <= 3 && (n_steps <= 0 || !capture_sizes || !sps)) return ORC_INVALID;
    if (mode >= 4 && !(conf_min == conf_min)) return ORC_INVALID;  // NaN cutoff
    if (K_cap < R) return ORC_CAPACITY;
    for (int i = 0; i < R * gamma; ++i) {
        if (!(c[i] >= 0.0f && c[i] <= 1.0f)) return ORC_DEVICE_INPUT;
        if (mode == 1 && !(c_hist[i] >= 0.0f && c_hist[i] <= 1.0f)) return ORC_DEVICE_INPUT;
    }

    auto survival = [&](const float* conf, float* out) {
        for (int r = 0; r < R; ++r) {
            float run = 1.0f;
            for (int k = 0; k < gamma; ++k) {
                run = (k == 0) ? conf[(size_t)r * gamma] : run * conf[(size_t)r * gamma + k];
                out[(size_t)r * gamma + k] = run;
            }
        }
    };
    // Candidate order: a descending, k ascending, r ascending.
    auto ordered = [&](const float* av) {
        std::vector<int> idx(R * gamma);
        for (int i = 0; i < R * gamma; ++i) idx[i] = i;
        std::sort(idx.begin(), idx.end(), [&](int x, int yv) {
            const float ax = av[x], ay = av[yv];
            if (ax != ay) return ax > ay;
            const int kx = x % gamma, ky = yv % gamma;
            if (kx != ky) return kx < ky;
            return x / gamma < yv / gamma;
        });
        return idx;
    };
    auto top_sum = [&](const float* av, const std::vector<int>& ord, int n) {
        double s = 0.0;
        for (int i = 0; i < n; ++i) s += (double)av[ord[i]];
        return s;
    };
    auto pad_rows = [&](int B) -> int {  // index of the smallest capture size >= B, -1 if none
        int best = -1;
        for (int i = 0; i < n_steps; ++i)
            if (capture_sizes[i] >= B && (best < 0 || capture_sizes[i] < capture_sizes[best])) best = i;
        return best;
    };

    survival(c, a);
    std::vector<int> ord = ordered(a);
    const int n_all = R * gamma;
    int n = 0;
    double gap = std::numeric_limits<double>::infinity();

    if (mode == 4 || mode == 5) {
        // eligible: each request's leading positions passing the cutoff; the
        // selection keeps the order above, restricted to eligible candidates
        std::vector<char> elig(n_all, 0);
        int n_elig = 0;
        for (int r = 0; r < R; ++r)
            for (int k = 0; k < gamma; ++k) {
                const float v = (mode == 4) ? c[(size_t)r * gamma + k] : a[(size_t)r * gamma + k];
                if (!(v >= conf_min)) break;
                elig[(size_t)r * gamma + k] = 1;
                ++n_elig;
            }
        std::vector<int> kept;
        for (int i : ord)
            if (elig[i]) kept.push_back(i);
        ord.swap(kept);
        n = std::min(n_elig, K_cap - R);
    } else if (mode == 0) {
        n = std::min(K_cap - R, n_all);
    } else if (mode == 1 || mode == 2) {
        std::vector<float> ah(n_all);
        const float* plan = a;
        std::vector<int> ord_h;
        if (mode == 1) { survival(c_hist, ah.data()); plan = ah.data(); ord_h = ordered(plan); }
        const std::vector<int>& po = (mode == 1) ? ord_h : ord;
        double best = -1.0, second = -1.0;
        int best_S = -1, best_n = 0;
        for (int i = 0; i < n_steps; ++i) {
            const int S = capture_sizes[i];
            if (S < R) continue;
            const int ni = std::min(std::min(S, K_cap) - R, n_all);
            const double th = (double)sps[i] * ((double)R + top_sum(plan, po, ni));
            if (best_S < 0 || th > best || (th == best && S < best_S)) {
                if (best_S >= 0) second = std::max(second, best);
                best = th; best_S = S; best_n = ni;
            } else {
                second = std::max(second, th);
            }
        }
        n = (best_S < 0) ? 0 : best_n;
        if (best_S >= 0 && second >= 0.0) gap = (best - second) / best;
    } else {
        const int p0 = pad_rows(R);
        if (p0 >= 0) {
            double theta = (double)sps[p0] * (double)R;
            double run = 0.0;
            while (n < n_all) {
                const int B = R + n + 1;
                if (B > K_cap) break;
                const int pi = pad_rows(B);
                if (pi < 0) break;
                const double next = (double)sps[pi] * ((double)R + run + (double)a[ord[n]]);
                const double g = std::fabs(next - theta) / std::max(next, theta);
                gap = std::min(gap, g);
                if (!(next > theta)) break;
                theta = next;
                run += (double)a[ord[n]];
                ++n;
            }
        }
    }

    for (int r = 0; r < R; ++r) l[r] = 0;
    for (int i = 0; i < n; ++i) l[ord[i] / gamma] += 1;
    cu_seqlens[0] = 0;
    for (int r = 0; r < R; ++r) cu_seqlens[r + 1] = cu_seqlens[r] + l[r] + 1;
    if (K_used) *K_used = R + n;
    if (theta_gap) *theta_gap = gap;
    return ORC_OK;
}

// A run of consecutive scheduling cycles ([EXPL] section 10: the physical
// capacity of cycle t comes from the confidences of cycle t - lag (two steps
// back in the paper's implementation), the top-K of cycle t's own survival
// fills it; section 15 lists the wasted verify work among the metrics to
// watch).  Every cycle is one orc_select_prefix call on c_seq[t]; in HISTORY
// mode its c_hist is c_seq[t - lag], and the first lag cycles, which have no
// history yet, use the capacity K_cap (FIXED).  With n_full[t][r] = the number
// of leading drafts of request r that the target would accept in cycle t (a
// property of the drafts, independent of how many are verified), the cycle's
// outcome is n_acc[r] = min(n_full[t][r], l[r]), and per cycle:
//   stats[t][0] = SPS(Bpad) * (R + sum of the selected a)   predicted Theta
//   stats[t][1] = SPS(Bpad) * (R + sum_r n_acc[r])          achieved Theta
//   stats[t][2] = sum_r n_acc[r]                            accepted drafts
//   stats[t][3] = sum_r (l[r] - n_acc[r])                   wasted verify rows
// with B = K_used physical rows and Bpad the smallest capture size >= B (SPS
// = 0 when none is; stats[t][1..3] are 0 without n_full).
int orc_plan_cycles(const float* c_seq, const int32_t* n_full, const int32_t* capture_sizes,
                    const float* sps, int n_steps, int K_cap, int mode, float conf_min, int lag,
                    int n_cycles, int R, int gamma, int32_t* l_seq, int32_t* K_seq, double* stats,
                    double* theta_gap) {
    if (n_cycles <= 0 || lag < 1 || R <= 0 || gamma <= 0) return ORC_INVALID;
    if (n_steps <= 0 || !capture_sizes || !sps) return ORC_INVALID;
    std::vector<float> a((size_t)R * gamma);
    std::vector<int32_t> cu(R + 1);
    int status = ORC_OK;
    for (int t = 0; t < n_cycles; ++t) {
        const float* ct = c_seq + (size_t)t * R * gamma;
        int m = mode;
        const float* hist = nullptr;
        if (mode == 1) {
            if (t >= lag) hist = c_seq + (size_t)(t - lag) * R * gamma;
            else m = 0;
        }
        int32_t K = 0;
        double gap = 0.0;
        int32_t* lt = l_seq + (size_t)t * R;
        const int st = orc_select_prefix(ct, hist, capture_sizes, sps, n_steps, K_cap, m, conf_min, R,
                                         gamma, a.data(), lt, cu.data(), &K, &gap);
        if (theta_gap) theta_gap[t] = gap;
        K_seq[t] = K;
        double* out = stats + (size_t)t * 4;
        out[0] = out[1] = out[2] = out[3] = 0.0;
        if (st != ORC_OK) { status = st; continue; }
        int best = -1;  // smallest capture size >= K
        for (int i = 0; i < n_steps; ++i)
            if (capture_sizes[i] >= K && (best < 0 || capture_sizes[i] < capture_sizes[best])) best = i;
        const double rate = best < 0 ? 0.0 : (double)sps[best];
        double sel = 0.0;
        long acc = 0, wasted = 0;
        for (int r = 0; r < R; ++r) {
            for (int k = 0; k < lt[r]; ++k) sel += (double)a[(size_t)r * gamma + k];
            if (n_full) {
                const int na = std::min((int)n_full[(size_t)t * R + r], (int)lt[r]);
                acc += na;
                wasted += lt[r] - na;
            }
        }
        out[0] = rate * ((double)R + sel);
        if (n_full) {
            out[1] = rate * ((double)R + (double)acc);
            out[2] = (double)acc;
            out[3] = (double)wasted;
        }
    }
    return status;
}

// Sequential temperature scaling of the confidence head ([EXPL] section 8:
// the per-position confidences are calibrated left to right by a post-hoc
// temperature so that their products are calibrated survival probabilities;
// the llama.cpp PR's "Future work" names the paper's Sequential Temperature
// Scaling calibration).  Position k is fitted on the samples that reached it
// (every earlier draft accepted), so c_k = sigmoid(z_k / tau_k) estimates the
// conditional acceptance rate the survival product multiplies.  With
// beta = 1/tau the negative log-likelihood of the labels y,
//   NLL(beta) = sum_i softplus(beta z_i) - y_i beta z_i,
// is convex; Newton's method from beta = 1 takes steps g / h with
//   g = sum_i (sigmoid(beta z_i) - y_i) z_i,  h = sum_i s_i (1 - s_i) z_i^2,
// halving beta instead whenever a step would leave (0, inf), for a fixed
// kFitIters iterations (the iterate has converged long before), and clamps
// beta to [1e-3, 1e3].  A position no sample reached keeps tau = 1.
// tau[k] = 1 / beta; nll[k] = NLL(beta) / count; count[k] = samples used.
static const int kFitIters = 60;

static double softplus(double x) { return x > 0.0 ? x + std::log1p(std::exp(-x)) : std::log1p(std::exp(x)); }
static double sigmoid(double x) { return x >= 0.0 ? 1.0 / (1.0 + std::exp(-x)) : std::exp(x) / (1.0 + std::exp(x)); }

int orc_fit_temperatures(const float* z, const uint8_t* accepted, int N, int gamma, float* tau,
                         double* nll, int32_t* count) {
    if (N <= 0 || gamma <= 0) return ORC_INVALID;
    for (int k = 0; k < gamma; ++k) {
        // the samples that reached position k
        std::vector<int> use;
        for (int i = 0; i < N; ++i) {
            bool reached = true;
            for (int j = 0; j < k; ++j)
                if (!accepted[(size_t)i * gamma + j]) { reached = false; break; }
            if (reached) use.push_back(i);
        }
        if (count) count[k] = (int32_t)use.size();
        if (use.empty()) { tau[k] = 1.0f; if (nll) nll[k] = 0.0; continue; }
        double beta = 1.0;
        for (int it = 0; it < kFitIters; ++it) {
            double g = 0.0, h = 0.0;
            for (int i : use) {
                const double zi = (double)z[(size_t)i * gamma + k];
                const double yi = accepted[(size_t)i * gamma + k] ? 1.0 : 0.0;
                const double si = sigmoid(beta * zi);
                g += (si - yi) * zi;
                h += si * (1.0 - si) * zi * zi;
            }
            if (!(h > 0.0)) break;
            const double next = beta - g / h;
            beta = (next > 0.0 && std::isfinite(next)) ? next : 0.5 * beta;
        }
        beta = std::min(1e3, std::max(1e-3, beta));
        double f = 0.0;
        for (int i : use) {
            const double zi = (double)z[(size_t)i * gamma + k];
            const double yi = accepted[(size_t)i * gamma + k] ? 1.0 : 0.0;
            f += softplus(beta * zi) - yi * beta * zi;
        }
        tau[k] = (float)(1.0 / beta);
        if (nll) nll[k] = f / (double)use.size();
    }
    return ORC_OK;
}

// Paged KV cache around one verify ([EXPL] section 11: the target's verify
// writes its candidate rows into temporary pages or block-table entries; after
// the first rejection only the accepted prefix is promoted to committed state
// and everything else -- the rejected candidates' K/V and their metadata -- is
// released or rolled back; section 15 lists leaked or double-freed temporary
// state among the failure classes).
//
// State: per request r its committed length kv_len[r] (tokens) and a block
// table of page ids (max_blocks per request; page b holds positions
// [b P, (b + 1) P)); the committed pages are entries 0 .. ceil(kv_len/P) - 1,
// the rest are -1.  Free pages form a stack free_pages[0 .. free_top).
//
// orc_kv_reserve: verify writes l[r] + 1 rows at positions kv_len .. kv_len + l,
// so request r needs need[r] = ceil((kv_len + l + 1) / P) - ceil(kv_len / P)
// more pages.  With T = sum need, the top T pages of the stack are handed out
// in request order (request r takes free_pages[free_top - T + o_r + i], o_r =
// need of the requests before it) into its next block-table entries, and
// free_top -= T.  If T > free_top, or a request would pass max_blocks, nothing
// changes and the call reports a capacity error.
//
// orc_kv_commit: request r keeps its committed prefix plus the accepted
// drafts' rows: kv_len' = kv_len + n_acc + 1 (n_acc in [0, l]; otherwise the
// request commits nothing, kv_len' = kv_len, and the call reports bad input).
// Pages ceil(kv_len'/P) .. ceil((kv_len + l + 1)/P) - 1 held only rejected rows:
// they go back on the stack in request order (request r's at free_top + o_r +
// i, o_r = pages released by the requests before it), their entries become
// -1, and free_top grows by the total.  Entries that hold no page (-1) are
// skipped; if the stack (pool_pages entries) could not take the pages, nothing
// changes and the call reports bad input.
static int ceil_div(int a, int b) { return (a + b - 1) / b; }

int orc_kv_reserve(const int32_t* kv_len, const int32_t* l, int R, int P, int32_t* block_table,
                   int max_blocks, int32_t* free_pages, int32_t* free_top, int pool_pages, int32_t* reserved) {
    if (R <= 0 || P <= 0 || max_blocks <= 0) return ORC_INVALID;
    if (*free_top < 0 || *free_top > pool_pages) return ORC_DEVICE_INPUT;
    std::vector<int> need(R);
    long total = 0;
    for (int r = 0; r < R; ++r) {
        if (kv_len[r] < 0 || l[r] < 0) return ORC_DEVICE_INPUT;
        const int have = ceil_div(kv_len[r], P), want = ceil_div(kv_len[r] + l[r] + 1, P);
        if (want > max_blocks) return ORC_CAPACITY;
        need[r] = want - have;
        total += need[r];
    }
    if (total > *free_top) return ORC_CAPACITY;
    const int base = *free_top - (int)total;
    int o = 0;
    for (int r = 0; r < R; ++r) {
        const int have = ceil_div(kv_len[r], P);
        for (int i = 0; i < need[r]; ++i)
            block_table[(size_t)r * max_blocks + have + i] = free_pages[base + o + i];
        if (reserved) reserved[r] = need[r];
        o += need[r];
    }
    *free_top = base;
    return ORC_OK;
}

int orc_kv_commit(int32_t* kv_len, const int32_t* l, const int32_t* n_acc, int R, int P,
                  int32_t* block_table, int max_blocks, int32_t* free_pages, int32_t* free_top,
                  int pool_pages) {
    if (R <= 0 || P <= 0 || max_blocks <= 0) return ORC_INVALID;
    int status = ORC_OK;
    auto span = [&](int r, int& keep, int& held, int& new_len) {
        if (kv_len[r] < 0 || l[r] < 0) { keep = held = 0; new_len = kv_len[r]; return; }  // unusable: untouched
        held = std::min(max_blocks, ceil_div(kv_len[r] + l[r] + 1, P));
        int committed = n_acc[r] + 1;
        if (n_acc[r] < 0 || n_acc[r] > l[r]) committed = 0;
        new_len = kv_len[r] + committed;
        keep = ceil_div(new_len, P);
    };
    long pushes = 0;
    for (int r = 0; r < R; ++r) {
        int keep, held, new_len;
        span(r, keep, held, new_len);
        for (int b = keep; b < held; ++b)
            if (block_table[(size_t)r * max_blocks + b] >= 0) ++pushes;
    }
    if (*free_top < 0 || *free_top + pushes > pool_pages) return ORC_DEVICE_INPUT;
    int top = *free_top;
    for (int r = 0; r < R; ++r) {
        int keep, held, new_len;
        span(r, keep, held, new_len);
        if (n_acc[r] < 0 || n_acc[r] > l[r] || kv_len[r] < 0 || l[r] < 0) status = ORC_DEVICE_INPUT;
        for (int b = keep; b < held; ++b) {
            int32_t& e = block_table[(size_t)r * max_blocks + b];
            if (e >= 0) free_pages[top++] = e;
            e = -1;
        }
        kv_len[r] = new_len;
    }
    *free_top = top;
    return status;
}

// Commit lengths ([EXPL] section 2: each cycle commits the accepted prefix
// plus one target-correct token; section 11: everything verified beyond it is
// rolled back).  commit_len = n_acc + 1, cu_commit = exclusive running sum,
// discard = l - n_acc (l NULL: every request verified gamma drafts).
int orc_commit_lengths(const int32_t* n_acc, const int32_t* l, int R, int gamma,
                       int32_t* commit_len, int32_t* cu_commit, int32_t* discard,
                       int32_t* total) {
    if (R <= 0 || gamma <= 0) return ORC_INVALID;
    int status = ORC_OK;
    cu_commit[0] = 0;
    for (int r = 0; r < R; ++r) {
        const int lr = l ? l[r] : gamma;
        const int na = n_acc[r];
        if (na < 0 || na > lr || lr > gamma) {
            status = ORC_DEVICE_INPUT;
            commit_len[r] = 0;
            discard[r] = 0;
        } else {
            commit_len[r] = na + 1;
            discard[r] = lr - na;
        }
        cu_commit[r + 1] = cu_commit[r] + commit_len[r];
    }
    if (total) *total = cu_commit[R];
    return status;
}

}  // extern "C"
