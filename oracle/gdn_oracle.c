/*
 * Gated DeltaNet recurrence -- CPU oracle (fp64).  TEST INFRASTRUCTURE.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load or run this file.  The GPU library never links it, never calls it and
 * shares no code, header, table or helper with it.
 *
 * What it computes: for every sequence and every value head, the token-by-token
 * recurrence of "Transformer by Hand, ch. 7 -- Gated DeltaNet: the
 * token-by-token recurrence" (section "The formula", and the four numbered
 * steps of the delta_rule listing in section "qwen/deltanet.py"):
 *
 *     S <- exp(g_t) * S                       1. decay
 *     p  = S^T k_t                            2. look the key up
 *     S <- S + k_t (beta_t (v_t - p))^T       3. write only the difference
 *     o_t = scale * S^T q_t                   4. read with the query
 *
 * S is a dk x dv table (row = key dimension), one per (sequence, value head),
 * kept in fp64 here.  Value head h reads query/key head floor(h / (Hv/Hqk)): the
 * repeat_interleave of the GatedDeltaNet shell in the same chapter.
 *
 * mode 1 ("plain add") replaces step 2-3 by S <- S + beta_t k_t v_t^T: ordinary
 * gated linear attention (the "without the subtraction" remark below the
 * formula; the Mamba2 row of the update-rule table on the learn-llm "linear
 * attention" page).  It exists only so tests can pin the oracle against the
 * closed-form sum of linear attention.
 *
 * normalize_qk: q and k are divided by sqrt(sum x^2 + 1e-6) first (the l2norm
 * call of delta_rule; its eps is not printed on the pages, 1e-6 is the reading
 * taken).  scale multiplies every output (delta_rule divides q by sqrt(dk); the
 * formula itself has no scale, so the default used by callers is 1).
 *
 * Layouts (row-major, contiguous): q, k [Ttot, Hqk, dk]; v [Ttot, Hv, dv];
 * g, beta [Ttot, Hv]; S0, S_final [num_seqs, Hv, dk, dv]; out [Ttot, Hv, dv].
 * Sequence i covers tokens [cu[i], cu[i+1]) and starts from S0[i] (zeros when
 * S0 is NULL).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One (sequence, value head) pair, tokens [t0, t1). */
static void run_pair(const double* q, const double* k, const double* v, const double* g,
                     const double* beta, const double* S0, double* out, double* S_final,
                     int64_t t0, int64_t t1, int h, int Hqk, int Hv, int dk, int dv,
                     double scale, int mode, int normalize_qk, double* S, double* p,
                     double* qn, double* kn) {
    const int group = Hv / Hqk;
    const int hk = h / group;
    const size_t sz = (size_t)dk * dv;
    if (S0) memcpy(S, S0, sz * sizeof(double));
    else memset(S, 0, sz * sizeof(double));

    for (int64_t t = t0; t < t1; ++t) {
        const double* qt = q + ((size_t)t * Hqk + hk) * dk;
        const double* kt = k + ((size_t)t * Hqk + hk) * dk;
        const double* vt = v + ((size_t)t * Hv + h) * dv;
        const double gt = g[(size_t)t * Hv + h];
        const double bt = beta[(size_t)t * Hv + h];
        double* ot = out + ((size_t)t * Hv + h) * dv;

        if (normalize_qk) {
            double sq = 0.0, sk = 0.0;
            for (int i = 0; i < dk; ++i) { sq += qt[i] * qt[i]; sk += kt[i] * kt[i]; }
            const double rq = 1.0 / sqrt(sq + 1e-6), rk = 1.0 / sqrt(sk + 1e-6);
            for (int i = 0; i < dk; ++i) { qn[i] = qt[i] * rq; kn[i] = kt[i] * rk; }
            qt = qn;
            kt = kn;
        }

        /* 1. decay */
        const double alpha = exp(gt);
        for (size_t e = 0; e < sz; ++e) S[e] *= alpha;

        if (mode == 0) {
            /* 2. p = S^T k */
            for (int j = 0; j < dv; ++j) p[j] = 0.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) p[j] += S[(size_t)i * dv + j] * kt[i];
            /* 3. S += k (beta (v - p))^T */
            for (int j = 0; j < dv; ++j) p[j] = bt * (vt[j] - p[j]);
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kt[i] * p[j];
        } else {
            /* plain add: S += beta k v^T */
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += bt * kt[i] * vt[j];
        }

        /* 4. o = scale * S^T q */
        for (int j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) ot[j] += S[(size_t)i * dv + j] * qt[i];
        for (int j = 0; j < dv; ++j) ot[j] *= scale;
    }
    if (S_final) memcpy(S_final, S, sz * sizeof(double));
}

/*
 * Returns 0 on success, -1 on a bad argument.  nthreads <= 0 uses the OpenMP
 * default.  Pairs (sequence, value head) are independent and run in parallel.
 */
int gdn_oracle_forward(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* S0, double* out, double* S_final,
                       const int64_t* cu, int num_seqs, int Hqk, int Hv, int dk, int dv,
                       double scale, int mode, int normalize_qk, int nthreads) {
    if (!q || !k || !v || !g || !beta || !out || !cu) return -1;
    if (num_seqs < 0 || Hqk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hqk != 0) return -1;
    if (mode != 0 && mode != 1) return -1;
    const int64_t pairs = (int64_t)num_seqs * Hv;
    const size_t sz = (size_t)dk * dv;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
#endif
    {
        double* S = (double*)malloc(sz * sizeof(double));
        double* p = (double*)malloc((size_t)dv * sizeof(double));
        double* qn = (double*)malloc((size_t)dk * sizeof(double));
        double* kn = (double*)malloc((size_t)dk * sizeof(double));
        const int ok = S && p && qn && kn;
        if (!ok) bad = 1;
        /* every thread reaches the work-sharing loop; one without buffers skips its pairs */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t pr = 0; pr < pairs; ++pr) {
            if (!ok) { bad = 1; continue; }
            const int i = (int)(pr / Hv), h = (int)(pr % Hv);
            const double* s0 = S0 ? S0 + ((size_t)i * Hv + h) * sz : NULL;
            double* sf = S_final ? S_final + ((size_t)i * Hv + h) * sz : NULL;
            run_pair(q, k, v, g, beta, s0, out, sf, cu[i], cu[i + 1], h, Hqk, Hv, dk, dv,
                     scale, mode, normalize_qk, S, p, qn, kn);
        }
        free(S);
        free(p);
        free(qn);
        free(kn);
    }
    return bad ? -1 : 0;
}
