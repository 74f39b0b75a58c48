/*
 * Kimi Delta Attention (KDA) CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the package's smoke() entry and bench.py's CPU-baseline leg use
 * this file.  The CUDA library never links, loads or calls it, and it shares
 * no code, header or constant with the library.
 *
 * What it computes is the plain definition of the KDA recurrence: a gated
 * delta rule with channel-wise decay.  Per (sequence, head), with a key-channel
 * by value-channel state S (dk x dv), for each token t of the sequence in order:
 *
 *     S <- Diag(exp g_t) . S                 decay, one factor per key channel
 *     r <- S^T k_t                           the state's prediction for key k_t
 *     S <- S + beta_t . k_t (v_t - r)^T      delta-rule write
 *     o_t <- S^T q_t                         read-out from the updated state
 *
 * which is S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
 * o_t = S_t^T q_t.  Sources: Kimi K3 report as summarised on the llm-atlas page
 * "K3_RESEARCH.md", question ledger Q04 (fixed-shape recurrent state with
 * channel-wise decay and delta-rule writes) and Q05 (the write first removes
 * the state's existing prediction for the current key).  The pages cite the
 * report's section 2.1 Eq. 1 without printing it; the form above is the gated
 * delta rule those two ledger entries describe.
 * Readings taken where the pages are silent: no 1/sqrt(dk) scaling of q, the
 * read-out uses the updated state, exp is the natural exponential, the decay is
 * applied before the delta correction, g is per key channel and beta per
 * (token, head).
 *
 * Arithmetic is fp64 throughout.  q/k/v are read in their storage type (fp32,
 * or bf16 given as raw 16-bit patterns) and widened exactly; g, beta and the
 * initial state are fp32 and widened exactly.
 *
 * Compile-time switch KDA_ORACLE_MUTANT (tests only) plants one deliberate
 * mistake so that the tests can show each pin catches it; the default build
 * defines no mutant.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef KDA_ORACLE_MUTANT
#define KDA_ORACLE_MUTANT 0
#endif

/* Exact widening of a bf16 bit pattern: it is the top half of an fp32. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, int is_bf16, size_t idx)
{
    if (is_bf16)
        return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    return (double)((const float*)base)[idx];
}

typedef struct {
    int32_t num_seqs, num_heads, dk, dv, is_bf16;
    const int32_t* cu_seqlens;
    const void *q, *k, *v;
    const float *g, *beta, *init_state;
    double *out, *final_state;
    int64_t next_unit;            /* shared work counter: unit = seq * H + head */
} job_t;

/* One (sequence, head): the token-by-token recurrence above. */
static void run_unit(const job_t* J, int64_t unit, double* S, double* kt, double* qt, double* r)
{
    const int32_t H = J->num_heads, dk = J->dk, dv = J->dv;
    const int32_t n = (int32_t)(unit / H), h = (int32_t)(unit % H);
    const size_t ss = (size_t)dk * dv;

    if (J->init_state) {
        const float* s0 = J->init_state + ((size_t)n * H + h) * ss;
        for (size_t i = 0; i < ss; ++i) S[i] = (double)s0[i];
    } else {
        for (size_t i = 0; i < ss; ++i) S[i] = 0.0;
    }

    for (int32_t t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
        const size_t th = (size_t)t * H + h;
        const float* gt = J->g + th * dk;
        const double bt = (double)J->beta[th];
        for (int32_t c = 0; c < dk; ++c) {
            kt[c] = load_elem(J->k, J->is_bf16, th * dk + c);
            qt[c] = load_elem(J->q, J->is_bf16, th * dk + c);
        }
#if KDA_ORACLE_MUTANT == 1
        /* mutant 1: read-out taken from the state before this token's update */
        for (int32_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int32_t c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * qt[c];
            J->out[th * dv + j] = acc;
        }
#endif
#if KDA_ORACLE_MUTANT != 2
        /* decay: row c of S is key channel c */
        for (int32_t c = 0; c < dk; ++c) {
            const double a = exp((double)gt[c]);
            double* row = S + (size_t)c * dv;
            for (int32_t j = 0; j < dv; ++j) row[j] *= a;
        }
#endif
        /* prediction r = S^T k */
        for (int32_t j = 0; j < dv; ++j) r[j] = 0.0;
        for (int32_t c = 0; c < dk; ++c) {
            const double* row = S + (size_t)c * dv;
#if KDA_ORACLE_MUTANT == 4
            /* mutant 4: transposed operand (S k instead of S^T k; valid only when dk == dv) */
            for (int32_t j = 0; j < dv; ++j) r[j] += S[(size_t)j * dv + c] * kt[c];
            (void)row;
#else
            for (int32_t j = 0; j < dv; ++j) r[j] += row[j] * kt[c];
#endif
        }
        /* delta-rule write S += beta k (v - r)^T */
        for (int32_t j = 0; j < dv; ++j) {
            const double vj = load_elem(J->v, J->is_bf16, th * dv + j);
#if KDA_ORACLE_MUTANT == 3
            r[j] = bt * (vj + r[j]);   /* mutant 3: sign of the correction flipped */
#elif KDA_ORACLE_MUTANT == 5
            r[j] = (vj - r[j]);        /* mutant 5: beta dropped */
#else
            r[j] = bt * (vj - r[j]);
#endif
        }
        for (int32_t c = 0; c < dk; ++c) {
            double* row = S + (size_t)c * dv;
            for (int32_t j = 0; j < dv; ++j) row[j] += kt[c] * r[j];
        }
#if KDA_ORACLE_MUTANT == 2
        /* mutant 2: decay applied after the delta correction */
        for (int32_t c = 0; c < dk; ++c) {
            const double a = exp((double)gt[c]);
            double* row = S + (size_t)c * dv;
            for (int32_t j = 0; j < dv; ++j) row[j] *= a;
        }
#endif
#if KDA_ORACLE_MUTANT != 1
        /* read-out o = S^T q */
        for (int32_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int32_t c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * qt[c];
            J->out[th * dv + j] = acc;
        }
#endif
    }
    if (J->final_state) {
        double* sf = J->final_state + ((size_t)n * H + h) * ss;
        memcpy(sf, S, ss * sizeof(double));
    }
}

static void* worker(void* arg)
{
    job_t* J = (job_t*)arg;
    const size_t ss = (size_t)J->dk * J->dv;
    double* S = (double*)malloc(ss * sizeof(double));
    double* kt = (double*)malloc((size_t)J->dk * sizeof(double));
    double* qt = (double*)malloc((size_t)J->dk * sizeof(double));
    double* r = (double*)malloc((size_t)J->dv * sizeof(double));
    const int64_t units = (int64_t)J->num_seqs * J->num_heads;
    if (S && kt && qt && r) {
        for (;;) {
            const int64_t u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
            if (u >= units) break;
            run_unit(J, u, S, kt, qt, r);
        }
    }
    free(S); free(kt); free(qt); free(r);
    return NULL;
}

/*
 * kda_oracle_recurrent -- fp64 reference for prefill (and for decode, which is
 * the same recurrence with sequences of one token).
 *
 * Layouts (host memory, contiguous, caller-owned):
 *   q, k [T, H, dk]; v [T, H, dv]: fp32, or bf16 as uint16 bit patterns when is_bf16;
 *   g [T, H, dk] fp32; beta [T, H] fp32; cu_seqlens [N+1] int32 (cu[0] = 0, non-decreasing);
 *   init_state [N, H, dk, dv] fp32 or NULL (zero state);
 *   out [T, H, dv] fp64; final_state [N, H, dk, dv] fp64 or NULL.
 * Uses num_threads POSIX threads (<= 0: one).  Returns 0, or -1 on a bad
 * argument or allocation failure.
 */
int kda_oracle_recurrent(int32_t num_seqs, const int32_t* cu_seqlens, int32_t num_heads,
                         int32_t dk, int32_t dv, int32_t is_bf16,
                         const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* init_state,
                         double* out, double* final_state, int32_t num_threads)
{
    if (num_seqs < 0 || num_heads <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
    if (cu_seqlens[0] != 0) return -1;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (cu_seqlens[num_seqs] > 0 && (!q || !k || !v || !g || !beta || !out)) return -1;

    job_t J;
    J.num_seqs = num_seqs; J.num_heads = num_heads; J.dk = dk; J.dv = dv; J.is_bf16 = is_bf16 ? 1 : 0;
    J.cu_seqlens = cu_seqlens; J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
    J.init_state = init_state; J.out = out; J.final_state = final_state; J.next_unit = 0;

    if (num_threads <= 1) {
        worker(&J);
        return 0;
    }
    pthread_t* tid = (pthread_t*)malloc((size_t)num_threads * sizeof(pthread_t));
    if (!tid) return -1;
    int started = 0;
    for (int i = 0; i < num_threads; ++i) {
        if (pthread_create(&tid[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    return 0;
}

/* Build identification so a test can tell which mutant (0 = none) it loaded. */
int kda_oracle_mutant(void) { return KDA_ORACLE_MUTANT; }
