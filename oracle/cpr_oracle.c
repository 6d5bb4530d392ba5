/*
 * CPU oracle for the Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, fp64 definition that the
 * CUDA path is checked against.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header, table or
 * helper with the CUDA library, and it never reads a value produced by the GPU.
 *
 * What the method computes (sources):
 *   - "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section
 *     "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet": CPR keeps the token
 *     recurrence as the main function, evaluates it in parallel across chunks, and
 *     decode resynchronises the hidden state every C tokens.
 *   - "SkyRL IsoExec: vLLM 与 Megatron 的 logprob 差 ...", section
 *     "Gated DeltaNet 的第三条路：chunkwise-parallel recurrent": training and prefill
 *     first compute the recurrent state at every chunk boundary, then evaluate the
 *     outputs inside each chunk with a parallel recurrent scan; decode uses the
 *     recurrent form and resynchronises every chunk_size tokens.
 *   - The pages name the layer (Gated DeltaNet) without printing its formula.  The
 *     formula used here is the standard gated delta rule (Yang, Kautz & Hatamizadeh,
 *     "Gated Delta Networks", ICLR 2025):
 *         S_t = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *         o_t = S_t q_t,      alpha_t = exp(g_t),
 *     with S a dv x dk matrix (row i = value index, column j = key index).
 *
 * In exact arithmetic CPR reaches the plain recurrence's result; it differs from it
 * only in rounding.  So the oracle is the plain recurrence, in fp64.
 *
 * Storage conventions shared with callers (all row-major, packed variable length):
 *   q, k      [T, H, dk]         v, o     [T, H, dv]         g, beta  [T, H]
 *   cu_seqlens int32 [n_seqs + 1], cu_seqlens[0] = 0, non-decreasing.
 *   a state   [dk, dv] per (sequence, head): element (j, i) holds S[i][j].
 *   state_in / state_out  [n_seqs, H, dk, dv];  state_in may be NULL (zero state).
 *   boundary  [n_chunks_total, H, dk, dv]: the state at the start of every chunk.  The
 *             chunk grid is anchored at each sequence's own position 0; sequence n owns
 *             ceil(L_n / C) chunks, numbered in packed order.  May be NULL.
 *
 * Functions that follow the pages' algorithm (oracle_gdn_chunked) implement the
 * chunk update in the algebraic form of the Gated Delta Networks paper (its chunkwise
 * "WY / UT transform" section), derived again in the comment above chunk_update().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted mistakes, compiled only into throw-away test builds (ORACLE_MUTANT=n) so
 * the test suite can show that its pins catch each of them.  0 = the real oracle. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

static int64_t n_chunks_of(int64_t len, int C) { return (len + C - 1) / C; }

int oracle_version(void) { return 1 + 100 * ORACLE_MUTANT; }

/* Total number of chunks of a packed batch (sum over sequences of ceil(L/C)). */
int64_t oracle_num_chunks(const int32_t* cu_seqlens, int n_seqs, int C)
{
    int64_t total = 0;
    for (int n = 0; n < n_seqs; ++n) total += n_chunks_of(cu_seqlens[n + 1] - cu_seqlens[n], C);
    return total;
}

/* Load a stored [dk, dv] state into the math layout S[i][j] (dv x dk). */
static void load_state(const double* stored, int dk, int dv, double* S)
{
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] = stored ? stored[(size_t)j * dv + i] : 0.0;
}

static void store_state(const double* S, int dk, int dv, double* stored)
{
    for (int j = 0; j < dk; ++j)
        for (int i = 0; i < dv; ++i) stored[(size_t)j * dv + i] = S[(size_t)i * dk + j];
}

/*
 * One token of the gated delta rule, written out from the formula
 *     S_t = alpha S (I - beta k k^T) + beta v k^T  =  alpha S - alpha beta (S k) k^T + beta v k^T,
 *     o   = S_t q.
 * S is dv x dk (math layout), updated in place; x is scratch of length dv.
 */
static void gdn_token(double* S, int dk, int dv, const double* k, const double* v, const double* q,
                      double g, double beta, double* x, double* o)
{
#if ORACLE_MUTANT == 6
    const double alpha = exp(-g);
#else
    const double alpha = exp(g);
#endif
    for (int i = 0; i < dv; ++i) { /* x = S_{t-1} k  (or its transpose, in a mutant) */
        double acc = 0.0;
#if ORACLE_MUTANT == 4
        for (int j = 0; j < dk; ++j) acc += S[(size_t)j * dk + i] * k[j];
#else
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * k[j];
#endif
        x[i] = acc;
    }
#if ORACLE_MUTANT == 3
    for (int i = 0; i < dv; ++i) { /* output from the state before the update */
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];
        o[i] = acc;
    }
#endif
    for (int i = 0; i < dv; ++i) {
        for (int j = 0; j < dk; ++j) {
            double s = S[(size_t)i * dk + j];
#if ORACLE_MUTANT == 1
            S[(size_t)i * dk + j] = alpha * s + alpha * beta * x[i] * k[j] + beta * v[i] * k[j];
#elif ORACLE_MUTANT == 2
            S[(size_t)i * dk + j] = s - alpha * beta * x[i] * k[j] + beta * v[i] * k[j];
#elif ORACLE_MUTANT == 5
            S[(size_t)i * dk + j] = alpha * s - alpha * x[i] * k[j] + v[i] * k[j];
#else
            S[(size_t)i * dk + j] = alpha * s - alpha * beta * x[i] * k[j] + beta * v[i] * k[j];
#endif
        }
    }
#if ORACLE_MUTANT != 3
    for (int i = 0; i < dv; ++i) { /* o = S_t q */
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];
        o[i] = acc;
    }
#endif
}

static int check_args(const int32_t* cu_seqlens, int n_seqs, int H, int dk, int dv, int C)
{
    if (!cu_seqlens || n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || C <= 0) return ORACLE_EINVAL;
    if (cu_seqlens[0] != 0) return ORACLE_EINVAL;
    for (int n = 0; n < n_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/*
 * The plain recurrence over a packed batch, token by token, in fp64.
 * Writes o for every token, the final state of every (sequence, head), and (if
 * boundary != NULL) the state at the start of every chunk of C tokens.
 * n_threads <= 0 lets OpenMP choose.
 */
int oracle_gdn_recurrent(const double* q, const double* k, const double* v, const double* g,
                         const double* beta, const int32_t* cu_seqlens, int n_seqs, int H, int dk,
                         int dv, int C, const double* state_in, double* o, double* state_out,
                         double* boundary, int n_threads)
{
    int rc = check_args(cu_seqlens, n_seqs, H, dk, dv, C);
    if (rc) return rc;
    int64_t* cu_chunks = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_seqs + 1));
    if (!cu_chunks) return ORACLE_ENOMEM;
    cu_chunks[0] = 0;
    for (int n = 0; n < n_seqs; ++n)
        cu_chunks[n + 1] = cu_chunks[n] + n_chunks_of(cu_seqlens[n + 1] - cu_seqlens[n], C);
    const size_t SS = (size_t)dk * dv;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int64_t p = 0; p < (int64_t)n_seqs * H; ++p) {
        const int n = (int)(p / H), h = (int)(p % H);
        double* S = (double*)malloc(sizeof(double) * SS);
        double* x = (double*)malloc(sizeof(double) * (size_t)dv);
        if (!S || !x) { failed = 1; free(S); free(x); continue; }
        load_state(state_in ? state_in + ((size_t)n * H + h) * SS : NULL, dk, dv, S);
        const int64_t t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - cu_seqlens[n];
        for (int64_t t = 0; t < L; ++t) {
            double* bnd = (boundary && t % C == 0)
                              ? boundary + ((size_t)(cu_chunks[n] + t / C) * H + h) * SS : NULL;
#if ORACLE_MUTANT != 7
            if (bnd) store_state(S, dk, dv, bnd); /* state before the chunk's first token */
#endif
            const size_t row = (size_t)(t0 + t) * H + h;
            gdn_token(S, dk, dv, k + row * dk, v + row * dv, q + row * dk, g[row], beta[row], x,
                      o + row * dv);
#if ORACLE_MUTANT == 7
            if (bnd) store_state(S, dk, dv, bnd); /* planted: one token too late */
#endif
        }
        if (state_out) store_state(S, dk, dv, state_out + ((size_t)n * H + h) * SS);
        free(S);
        free(x);
    }
    free(cu_chunks);
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* C = A (m x p) * B (p x r), all math-layout row-major doubles. */
static void matmul(const double* A, const double* B, double* Cm, int m, int p, int r)
{
    for (int i = 0; i < m; ++i)
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int l = 0; l < p; ++l) acc += A[(size_t)i * p + l] * B[(size_t)l * r + j];
            Cm[(size_t)i * r + j] = acc;
        }
}

/*
 * Brute force for one (sequence, head), for tiny sizes only.  It never runs the
 * recurrence: it materialises the per-token transition matrices
 *     M_t = alpha_t (I - beta_t k_t k_t^T)          (dk x dk)
 * and evaluates, for every t from scratch,
 *     S_t = S_0 M_0 M_1 ... M_t + sum_{s<=t} beta_s v_s k_s^T M_{s+1} ... M_t,
 *     o_t = S_t q_t.
 * Layouts: q, k [T, dk]; v [T, dv]; g, beta [T]; S0 and ST stored [dk, dv]; o [T, dv].
 */
int oracle_gdn_bruteforce(const double* q, const double* k, const double* v, const double* g,
                          const double* beta, int T, int dk, int dv, const double* S0, double* o,
                          double* ST)
{
    if (T < 0 || dk <= 0 || dv <= 0) return ORACLE_EINVAL;
    const size_t KK = (size_t)dk * dk, VK = (size_t)dv * dk;
    double* M = (double*)malloc(sizeof(double) * KK * (size_t)(T > 0 ? T : 1));
    double* P = (double*)malloc(sizeof(double) * KK);
    double* tmp = (double*)malloc(sizeof(double) * KK);
    double* S = (double*)malloc(sizeof(double) * VK);
    double* S0m = (double*)malloc(sizeof(double) * VK);
    double* term = (double*)malloc(sizeof(double) * VK);
    double* term2 = (double*)malloc(sizeof(double) * VK);
    if (!M || !P || !tmp || !S || !S0m || !term || !term2) {
        free(M); free(P); free(tmp); free(S); free(S0m); free(term); free(term2);
        return ORACLE_ENOMEM;
    }
    load_state(S0, dk, dv, S0m);
    for (int t = 0; t < T; ++t) {
        const double a = exp(g[t]);
        for (int r = 0; r < dk; ++r)
            for (int c = 0; c < dk; ++c)
                M[(size_t)t * KK + (size_t)r * dk + c] =
                    a * ((r == c ? 1.0 : 0.0) - beta[t] * k[(size_t)t * dk + r] * k[(size_t)t * dk + c]);
    }
    if (T == 0) memcpy(S, S0m, sizeof(double) * VK);
    for (int t = 0; t < T; ++t) {
        /* S_t = S_0 * (M_0 ... M_t) */
        for (int r = 0; r < dk; ++r)
            for (int c = 0; c < dk; ++c) P[(size_t)r * dk + c] = (r == c) ? 1.0 : 0.0;
        for (int s = 0; s <= t; ++s) {
            matmul(P, M + (size_t)s * KK, tmp, dk, dk, dk);
            memcpy(P, tmp, sizeof(double) * KK);
        }
        matmul(S0m, P, S, dv, dk, dk);
        /* + sum_{s<=t} beta_s v_s k_s^T (M_{s+1} ... M_t) */
        for (int s = 0; s <= t; ++s) {
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j)
                    term[(size_t)i * dk + j] = beta[s] * v[(size_t)s * dv + i] * k[(size_t)s * dk + j];
            for (int u = s + 1; u <= t; ++u) {
                matmul(term, M + (size_t)u * KK, term2, dv, dk, dk);
                memcpy(term, term2, sizeof(double) * VK);
            }
            for (size_t e = 0; e < VK; ++e) S[e] += term[e];
        }
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[(size_t)t * dk + j];
            o[(size_t)t * dv + i] = acc;
        }
    }
    if (ST) store_state(S, dk, dv, ST);
    free(M); free(P); free(tmp); free(S); free(S0m); free(term); free(term2);
    return ORACLE_OK;
}

/*
 * The chunk update U(S_b, chunk) in fp64, for one full chunk of n tokens r = 0..n-1.
 *
 * Derivation (gated delta rule, chunkwise form of the Gated Delta Networks paper).
 * Inside the chunk write S_r = alpha_r S_{r-1} + delta_r k_r^T with
 *     delta_r = beta_r (v_r - alpha_r S_{r-1} k_r),      S_{-1} = S_b.
 * With G_r = g_0 + ... + g_r (so e^{G_r} = alpha_0 ... alpha_r), unrolling gives
 *     S_r = e^{G_r} S_b + sum_{i<=r} e^{G_r - G_i} delta_i k_i^T,
 * and substituting S_{r-1} into delta_r:
 *     delta_r + sum_{i<r} A_ri delta_i = beta_r v_r - beta_r e^{G_r} S_b k_r,
 *     A_ri = beta_r e^{G_r - G_i} (k_r . k_i)        (i < r; A is strictly lower).
 * So with T = (I + A)^{-1}:
 *     Delta = U~ - W S_b^T,   U~ = T diag(beta) V,   W = T diag(beta e^{G}) K,
 *     S_new = e^{G_{n-1}} S_b + sum_r e^{G_{n-1} - G_r} delta_r k_r^T.
 * T is applied by forward substitution (row r of W and U~ from rows i < r).
 *
 * kc [n, dk], vc [n, dv], gc, bc [n] are the chunk's tokens; Sb and Snew are math layout.
 */
static int chunk_update(const double* Sb, const double* kc, const double* vc, const double* gc,
                        const double* bc, int n, int dk, int dv, double* Snew)
{
    double* G = (double*)malloc(sizeof(double) * (size_t)n);
    double* A = (double*)malloc(sizeof(double) * (size_t)n * n);
    double* W = (double*)malloc(sizeof(double) * (size_t)n * dk);
    double* U = (double*)malloc(sizeof(double) * (size_t)n * dv);
    double* D = (double*)malloc(sizeof(double) * (size_t)n * dv);
    if (!G || !A || !W || !U || !D) { free(G); free(A); free(W); free(U); free(D); return ORACLE_ENOMEM; }
    double acc = 0.0;
    for (int r = 0; r < n; ++r) { acc += gc[r]; G[r] = acc; }
    for (int r = 0; r < n; ++r)
        for (int i = 0; i < n; ++i) {
            double a = 0.0;
            if (i < r) {
                double kk = 0.0;
                for (int j = 0; j < dk; ++j) kk += kc[(size_t)r * dk + j] * kc[(size_t)i * dk + j];
#if ORACLE_MUTANT == 8
                a = bc[r] * exp(G[i] - G[r]) * kk;
#else
                a = bc[r] * exp(G[r] - G[i]) * kk;
#endif
            }
            A[(size_t)r * n + i] = a;
        }
    /* forward substitution: (I + A) W = diag(beta e^G) K,  (I + A) U~ = diag(beta) V */
    for (int r = 0; r < n; ++r) {
        for (int j = 0; j < dk; ++j) {
            double w = bc[r] * exp(G[r]) * kc[(size_t)r * dk + j];
            for (int i = 0; i < r; ++i) w -= A[(size_t)r * n + i] * W[(size_t)i * dk + j];
            W[(size_t)r * dk + j] = w;
        }
        for (int c = 0; c < dv; ++c) {
            double u = bc[r] * vc[(size_t)r * dv + c];
            for (int i = 0; i < r; ++i) u -= A[(size_t)r * n + i] * U[(size_t)i * dv + c];
            U[(size_t)r * dv + c] = u;
        }
    }
    /* Delta = U~ - W S_b^T   (row r, column c = value index) */
    for (int r = 0; r < n; ++r)
        for (int c = 0; c < dv; ++c) {
            double ws = 0.0;
            for (int j = 0; j < dk; ++j) ws += W[(size_t)r * dk + j] * Sb[(size_t)c * dk + j];
            D[(size_t)r * dv + c] = U[(size_t)r * dv + c] - ws;
        }
    /* S_new = e^{G_{n-1}} S_b + sum_r e^{G_{n-1} - G_r} delta_r k_r^T */
    const double gamma = exp(G[n - 1]);
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) {
            double s = gamma * Sb[(size_t)i * dk + j];
            for (int r = 0; r < n; ++r) {
#if ORACLE_MUTANT == 9
                const double d = 1.0;
#else
                const double d = exp(G[n - 1] - G[r]);
#endif
                s += d * D[(size_t)r * dv + i] * kc[(size_t)r * dk + j];
            }
            Snew[(size_t)i * dk + j] = s;
        }
    free(G); free(A); free(W); free(U); free(D);
    return ORACLE_OK;
}

/*
 * The CPR schedule itself, in fp64: for every (sequence, head) and every chunk,
 * record the boundary state, evaluate the chunk's outputs by the token recurrence
 * from that boundary state, and obtain the next boundary state with the chunk update
 * U (full chunks) or, for a sequence's final partial chunk, keep the stepped state.
 * Same arguments and layouts as oracle_gdn_recurrent.  In exact arithmetic the two
 * agree; in fp64 they agree to rounding, which is what the tests check.
 */
int oracle_gdn_chunked(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const int32_t* cu_seqlens, int n_seqs, int H, int dk,
                       int dv, int C, const double* state_in, double* o, double* state_out,
                       double* boundary, int n_threads)
{
    int rc = check_args(cu_seqlens, n_seqs, H, dk, dv, C);
    if (rc) return rc;
    int64_t* cu_chunks = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_seqs + 1));
    if (!cu_chunks) return ORACLE_ENOMEM;
    cu_chunks[0] = 0;
    for (int n = 0; n < n_seqs; ++n)
        cu_chunks[n + 1] = cu_chunks[n] + n_chunks_of(cu_seqlens[n + 1] - cu_seqlens[n], C);
    const size_t SS = (size_t)dk * dv;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int64_t p = 0; p < (int64_t)n_seqs * H; ++p) {
        const int n = (int)(p / H), h = (int)(p % H);
        double* Sb = (double*)malloc(sizeof(double) * SS);
        double* S = (double*)malloc(sizeof(double) * SS);
        double* x = (double*)malloc(sizeof(double) * (size_t)dv);
        double* kc = (double*)malloc(sizeof(double) * (size_t)C * dk);
        double* vc = (double*)malloc(sizeof(double) * (size_t)C * dv);
        double* gc = (double*)malloc(sizeof(double) * (size_t)C);
        double* bc = (double*)malloc(sizeof(double) * (size_t)C);
        if (!Sb || !S || !x || !kc || !vc || !gc || !bc) {
            failed = 1;
            free(Sb); free(S); free(x); free(kc); free(vc); free(gc); free(bc);
            continue;
        }
        load_state(state_in ? state_in + ((size_t)n * H + h) * SS : NULL, dk, dv, Sb);
        const int64_t t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - cu_seqlens[n];
        for (int64_t j = 0; j * C < L; ++j) {
            const int64_t start = j * C;
            const int len = (int)((L - start) < C ? (L - start) : C);
            if (boundary) store_state(Sb, dk, dv, boundary + ((size_t)(cu_chunks[n] + j) * H + h) * SS);
            memcpy(S, Sb, sizeof(double) * SS);
            for (int r = 0; r < len; ++r) {
                const size_t row = (size_t)(t0 + start + r) * H + h;
                gdn_token(S, dk, dv, k + row * dk, v + row * dv, q + row * dk, g[row], beta[row], x,
                          o + row * dv);
                memcpy(kc + (size_t)r * dk, k + row * dk, sizeof(double) * dk);
                memcpy(vc + (size_t)r * dv, v + row * dv, sizeof(double) * dv);
                gc[r] = g[row];
                bc[r] = beta[row];
            }
            if (len == C) {
                if (chunk_update(Sb, kc, vc, gc, bc, C, dk, dv, S)) { failed = 1; break; }
            }
#if ORACLE_MUTANT == 10
            if (len < C) continue; /* planted: final partial chunk keeps its boundary state */
#endif
            memcpy(Sb, S, sizeof(double) * SS);
        }
        if (state_out) store_state(Sb, dk, dv, state_out + ((size_t)n * H + h) * SS);
        free(Sb); free(S); free(x); free(kc); free(vc); free(gc); free(bc);
    }
    free(cu_chunks);
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* Number of OpenMP threads the oracle uses by default (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
