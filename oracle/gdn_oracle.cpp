// Gated DeltaNet CPU oracle -- TEST INFRASTRUCTURE ONLY.
//
// Plain, slow, fp64 reference for the gated delta rule.  It is used by the
// test suite, by the smoke check and by the benchmark's CPU-baseline leg to
// check the CUDA library; the library never calls it, links it or shares
// code with it.
//
// What it computes (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配",
// section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet", which names
// Gated DeltaNet and its recurrent decode form; the per-token update is the
// gated delta rule):
//
//     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
//     o_t = S_t (scale * q_t),        alpha_t = exp(g_t)
//
// S_t is d_v x d_k.  The public layout stores H = S^T (d_k x d_v), so
// h0 / hT are [n_seq, H, d_k, d_v].  Token-major tensors:
//     q, k [n_tok, H, d_k];  v, o [n_tok, H, d_v];  g, beta [n_tok, H].
// Sequences are packed by cu_seqlens (n_seq + 1 int32 offsets); every
// (sequence, head) pair is an independent recurrence.
//
// The forward is the token-by-token recurrence in fp64.  The backward is a
// hand-derived reverse recurrence (adjoint of each token update), with the
// forward states recomputed segment by segment from checkpoints taken every
// `seg` tokens.  Written from the recurrence above; no chunking, no blocking,
// no reordering beyond the definition.
//
// Parity pins for both functions live in tests/test_oracle_*.py.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Problem {
    int n_seq;
    const int32_t* cu;
    int H, dk, dv;
    double scale;
    const double *q, *k, *v, *g, *beta, *h0;
};

// S stored row-major: S[i * dk + j], i over d_v, j over d_k.
inline void load_state(const Problem& P, int b, int h, std::vector<double>& S) {
    S.assign((size_t)P.dv * P.dk, 0.0);
    if (!P.h0) return;
    const double* H0 = P.h0 + ((size_t)b * P.H + h) * P.dk * P.dv;
    for (int j = 0; j < P.dk; ++j)
        for (int i = 0; i < P.dv; ++i) S[(size_t)i * P.dk + j] = H0[(size_t)j * P.dv + i];
}

// One token of the recurrence: S <- alpha S (I - beta k k^T) + beta v k^T,
// written as S <- alpha S;  u = S k;  S <- S + beta (v - u) k^T.
inline void token_update(const Problem& P, size_t t, int h, std::vector<double>& S,
                         std::vector<double>& u) {
    const int dk = P.dk, dv = P.dv;
    const double alpha = std::exp(P.g[t * P.H + h]);
    const double bt = P.beta[t * P.H + h];
    const double* kt = P.k + (t * P.H + h) * dk;
    const double* vt = P.v + (t * P.H + h) * dv;
    for (auto& x : S) x *= alpha;
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * kt[j];
        u[i] = acc;
    }
    for (int i = 0; i < dv; ++i) {
        const double e = bt * (vt[i] - u[i]);
        for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += e * kt[j];
    }
}

template <class F>
void parallel_units(int n_units, int n_threads, F&& fn) {
    if (n_threads <= 0) n_threads = (int)std::thread::hardware_concurrency();
    if (n_threads <= 0) n_threads = 1;
    if (n_threads > n_units) n_threads = n_units > 0 ? n_units : 1;
    std::atomic<int> next{0};
    auto worker = [&]() {
        for (;;) {
            int u = next.fetch_add(1);
            if (u >= n_units) break;
            fn(u);
        }
    };
    std::vector<std::thread> pool;
    for (int i = 1; i < n_threads; ++i) pool.emplace_back(worker);
    worker();
    for (auto& th : pool) th.join();
}

bool check_cu(const Problem& P) {
    if (P.n_seq < 0 || P.H <= 0 || P.dk <= 0 || P.dv <= 0) return false;
    if (P.cu[0] != 0) return false;
    for (int b = 0; b < P.n_seq; ++b)
        if (P.cu[b + 1] < P.cu[b]) return false;
    return true;
}

}  // namespace

extern "C" {

// Forward: o (required), hT (nullable).  h0 nullable (zeros).
// Returns 0 on success, 1 on bad arguments.
int oracle_gdn_fwd(int n_seq, const int32_t* cu_seqlens, int H, int dk, int dv, double scale,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta, const double* h0, double* o, double* hT, int n_threads) {
    Problem P{n_seq, cu_seqlens, H, dk, dv, scale, q, k, v, g, beta, h0};
    if (!check_cu(P) || !o) return 1;
    parallel_units(n_seq * H, n_threads, [&](int unit) {
        const int b = unit / H, h = unit % H;
        std::vector<double> S, u(dv);
        load_state(P, b, h, S);
        for (size_t t = (size_t)cu_seqlens[b]; t < (size_t)cu_seqlens[b + 1]; ++t) {
            token_update(P, t, h, S, u);
            const double* qt = q + (t * H + h) * dk;
            double* ot = o + (t * H + h) * dv;
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qt[j];
                ot[i] = scale * acc;
            }
        }
        if (hT) {
            double* HT = hT + ((size_t)b * H + h) * dk * dv;
            for (int j = 0; j < dk; ++j)
                for (int i = 0; i < dv; ++i) HT[(size_t)j * dv + i] = S[(size_t)i * dk + j];
        }
    });
    return 0;
}

// Backward of the forward above for the loss  sum(dO * o) + sum(dHT * hT).
// Outputs dq, dk, dv [tokens], dg, dbeta [tokens], dh0 [n_seq, H, d_k, d_v]
// (all required).  dHT nullable (zero).  `seg` is the checkpoint spacing
// (tokens) for recomputing forward states; it does not change the result
// beyond fp64 rounding of identical operations (states are recomputed by the
// same token update).
//
// Reverse step for token t, with Sh = dL/dS_t accumulated from later tokens
// (derived from the token update; S_a = alpha S_{t-1}, e = v - S_a k):
//     Sh    += scale * do_t q_t^T
//     dq_t   = scale * S_t^T do_t
//     sk     = Sh k_t
//     dv_t   = beta sk
//     dbeta  = e . sk
//     dk_t   = beta Sh^T e - alpha beta S_{t-1}^T sk
//     dalpha = <Sh, S_{t-1}> - beta sk . (S_{t-1} k_t)
//     dg_t   = alpha dalpha
//     Sh     = alpha (Sh - beta sk k_t^T)
// and dh0 = Sh^T after the first token.
int oracle_gdn_bwd(int n_seq, const int32_t* cu_seqlens, int H, int dk, int dv, double scale,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta, const double* h0, const double* dO, const double* dHT,
                   double* dq, double* dk_out, double* dv_out, double* dg, double* dbeta,
                   double* dh0, int seg, int n_threads) {
    Problem P{n_seq, cu_seqlens, H, dk, dv, scale, q, k, v, g, beta, h0};
    if (!check_cu(P) || !dO || !dq || !dk_out || !dv_out || !dg || !dbeta || !dh0) return 1;
    if (seg <= 0) seg = 64;
    parallel_units(n_seq * H, n_threads, [&](int unit) {
        const int b = unit / H, h = unit % H;
        const size_t t0 = (size_t)cu_seqlens[b], t1 = (size_t)cu_seqlens[b + 1];
        const size_t T = t1 - t0;
        const size_t SS = (size_t)dv * dk;
        std::vector<double> S, u(dv);
        load_state(P, b, h, S);
        // checkpoints: state before token t0 + c*seg
        const size_t n_seg = (T + seg - 1) / seg;
        std::vector<double> ckpt(n_seg * SS);
        for (size_t c = 0; c < n_seg; ++c) {
            std::memcpy(&ckpt[c * SS], S.data(), SS * sizeof(double));
            const size_t a = t0 + c * seg, e = std::min(t1, a + seg);
            for (size_t t = a; t < e; ++t) token_update(P, t, h, S, u);
        }
        // adjoint of the final state
        std::vector<double> Sh(SS, 0.0);
        if (dHT) {
            const double* D = dHT + ((size_t)b * H + h) * dk * dv;
            for (int j = 0; j < dk; ++j)
                for (int i = 0; i < dv; ++i) Sh[(size_t)i * dk + j] = D[(size_t)j * dv + i];
        }
        std::vector<double> states((size_t)(seg + 1) * SS);
        std::vector<double> sk(dv), w(dv), e(dv);
        for (size_t c = n_seg; c-- > 0;) {
            const size_t a = t0 + c * seg, end = std::min(t1, a + seg);
            // states[i] = S after (a - t0 + i) tokens
            std::memcpy(&states[0], &ckpt[c * SS], SS * sizeof(double));
            S.assign(states.begin(), states.begin() + SS);
            for (size_t t = a; t < end; ++t) {
                token_update(P, t, h, S, u);
                std::memcpy(&states[(t - a + 1) * SS], S.data(), SS * sizeof(double));
            }
            for (size_t t = end; t-- > a;) {
                const double* Sprev = &states[(t - a) * SS];
                const double* Scur = &states[(t - a + 1) * SS];
                const double* qt = q + (t * H + h) * dk;
                const double* kt = k + (t * H + h) * dk;
                const double* vt = v + (t * H + h) * dv;
                const double* dot = dO + (t * H + h) * dv;
                const double alpha = std::exp(g[t * H + h]);
                const double bt = beta[t * H + h];
                // o_t = scale * S_t q_t
                for (int i = 0; i < dv; ++i)
                    for (int j = 0; j < dk; ++j) Sh[(size_t)i * dk + j] += scale * dot[i] * qt[j];
                double* dqt = dq + (t * H + h) * dk;
                for (int j = 0; j < dk; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dv; ++i) acc += Scur[(size_t)i * dk + j] * dot[i];
                    dqt[j] = scale * acc;
                }
                for (int i = 0; i < dv; ++i) {
                    double a1 = 0.0, a2 = 0.0;
                    for (int j = 0; j < dk; ++j) {
                        a1 += Sprev[(size_t)i * dk + j] * kt[j];
                        a2 += Sh[(size_t)i * dk + j] * kt[j];
                    }
                    w[i] = a1;
                    sk[i] = a2;
                    e[i] = vt[i] - alpha * a1;
                }
                double* dvt = dv_out + (t * H + h) * dv;
                double db = 0.0, skw = 0.0;
                for (int i = 0; i < dv; ++i) {
                    dvt[i] = bt * sk[i];
                    db += e[i] * sk[i];
                    skw += sk[i] * w[i];
                }
                dbeta[t * H + h] = db;
                double* dkt = dk_out + (t * H + h) * dk;
                for (int j = 0; j < dk; ++j) {
                    double a1 = 0.0, a2 = 0.0;
                    for (int i = 0; i < dv; ++i) {
                        a1 += Sh[(size_t)i * dk + j] * e[i];
                        a2 += Sprev[(size_t)i * dk + j] * sk[i];
                    }
                    dkt[j] = bt * a1 - alpha * bt * a2;
                }
                double inner = 0.0;
                for (size_t x = 0; x < SS; ++x) inner += Sh[x] * Sprev[x];
                const double dalpha = inner - bt * skw;
                dg[t * H + h] = alpha * dalpha;
                for (int i = 0; i < dv; ++i)
                    for (int j = 0; j < dk; ++j) {
                        double& s = Sh[(size_t)i * dk + j];
                        s = alpha * (s - bt * sk[i] * kt[j]);
                    }
            }
        }
        double* D0 = dh0 + ((size_t)b * H + h) * dk * dv;
        for (int j = 0; j < dk; ++j)
            for (int i = 0; i < dv; ++i) D0[(size_t)j * dv + i] = Sh[(size_t)i * dk + j];
    });
    return 0;
}

}  // extern "C"
