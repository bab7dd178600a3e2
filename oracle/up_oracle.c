/*
 * up_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow fp64 CPU restatement of UniPrefill's block-wise dynamic
 * sparsification hot path: block scoring from the last n queries, top-p block
 * selection, and compaction of the kept tokens (sparsity propagation).
 *
 * Sources (web pages; none of them prints code):
 *   [UP]  "UniPrefill: 블록 단위 동적 희소화를 통한 범용적 롱 컨텍스트 프리필 가속화"
 *         (aitrends.kr overview): the drop-criterion paragraph, the block-wise
 *         importance-estimation paragraph, the top-p selection paragraph, the
 *         sparsity-propagation paragraph and the system-integration paragraph.
 *   [UPA] "UniPrefill: Universal Long-Context Prefill Acceleration via Block-wise
 *         Dynamic Sparsification", abstract (chatpaper.ai): the operator works on
 *         continuously batched (varlen) sequences.
 *   [CP]  Ultralytics glossary "Chunked Prefill", section "how chunked prefill
 *         works": the causal mask is taken over absolute positions.
 *
 * Only tests/, the package's smoke() entry and bench.py's CPU-baseline leg use
 * this file. It shares no code, header, table or helper with the CUDA library;
 * neither includes nor links the other.
 *
 * Readings where the pages are silent (each restated where it is used):
 *   - the softmax is per query over its visible keys; probabilities are then
 *     summed into blocks (no second softmax over blocks);
 *   - a block's score is the SUM of its tokens' mass, averaged over queries and
 *     heads, so the scores of one sequence sum to 1;
 *   - key i is visible to the query at absolute position a iff i <= a;
 *   - n_s = min(n, L_s); logits are q.k / sqrt(d), no softcap;
 *   - query head h reads KV head h / (Hq / Hk) (contiguous GQA groups);
 *   - top-p keeps the minimal score-sorted prefix whose cumulative mass reaches
 *     p, including the crossing block; p >= 1 keeps every block; ties go to the
 *     lower block index; cumulative sums are fp64;
 *   - top-k keeps the first min(k, nb) blocks of the same ranking; the
 *     optional keep-last step also keeps each sequence's last block;
 *   - compaction keeps ascending original order; positions are gathered, not
 *     renumbered.
 *
 * Pins (tests/test_oracle_pins.py): closed form for q == 0, a hand-worked
 * two-key softmax, fp64 torch.softmax on dense tiny cases, sum-to-one, the
 * G = 1 and G >= L special cases, GQA == MHA with repeated KV heads,
 * hand-enumerated and brute-force top-p and top-k sets, the keep-last step,
 * and compaction invariants.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> fp64 is exact: a bf16 value is the top 16 bits of an fp32 value. */
static double orc_bf16(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Token mass.                                                               */
/* [UP] block-wise importance estimation: the last n queries are dotted with  */
/* all N keys; [UP] drop criterion: a token matters through its softmax      */
/* probability.  For query head h and each of the last n_s queries t, at     */
/* absolute position a_t = L - n_s + t:                                       */
/*     z_i = (q_{t,h} . k_{i,j}) / sqrt(d)  for i <= a_t,  j = h / (Hq/Hk)     */
/*     P_i = exp(z_i - m) / sum_{i' <= a_t} exp(z_i' - m),  m = max_i z_i      */
/* and T_h[i] = sum_t P_i.  The token mass of the sequence is                 */
/*     T[i] = (sum_h T_h[i]) / (n_s * Hq),                                    */
/* heads merged in order h = 0 .. Hq-1, so the result does not depend on the  */
/* number of threads.                                                        */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;  /* q_last rows of this sequence: [n_s, Hq, d] */
    const uint16_t *k;  /* keys of this sequence: [L, Hk, d] */
    int L, ns, Hq, Hk, d;
    double *Th;         /* [Hq, L] per-head mass */
    int h_begin, h_step;
} orc_head_job;

static void *orc_head_worker(void *arg)
{
    orc_head_job *jb = (orc_head_job *)arg;
    const int L = jb->L, ns = jb->ns, Hq = jb->Hq, Hk = jb->Hk, d = jb->d;
    const int group = Hq / Hk;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    double *z = (double *)malloc(sizeof(double) * (size_t)L);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
    for (int h = jb->h_begin; h < Hq; h += jb->h_step) {
        const int j = h / group;
        double *T = jb->Th + (size_t)h * (size_t)L;
        for (int i = 0; i < L; ++i) T[i] = 0.0;
        for (int t = 0; t < ns; ++t) {
            const int a = L - ns + t; /* absolute position of this query */
            const uint16_t *qp = jb->q + ((size_t)t * Hq + h) * (size_t)d;
            for (int c = 0; c < d; ++c) qrow[c] = orc_bf16(qp[c]);
            double m = -INFINITY;
            for (int i = 0; i <= a; ++i) {
                const uint16_t *kp = jb->k + ((size_t)i * Hk + j) * (size_t)d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += qrow[c] * orc_bf16(kp[c]);
                z[i] = dot * inv_sqrt_d;
                if (z[i] > m) m = z[i];
            }
            double S = 0.0;
            for (int i = 0; i <= a; ++i) S += exp(z[i] - m);
            for (int i = 0; i <= a; ++i) T[i] += exp(z[i] - m) / S;
        }
    }
    free(qrow);
    free(z);
    return NULL;
}

/* mass[total_tokens] receives T for every token of every sequence.
 * q_last is [sum_s n_s, Hq, d] (the last n_s tokens of each sequence, packed
 * in sequence order); k is [total_tokens, Hk, d]; both hold bf16 bit patterns.
 * Returns 0 on success, -1 on a bad argument or allocation failure. */
int orc_token_mass(const uint16_t *q_last, const uint16_t *k, const int32_t *cu_seqlens,
                   int num_seqs, int Hq, int Hk, int d, int n, double *mass, int nthreads)
{
    if (num_seqs < 0 || Hq < 1 || Hk < 1 || Hq % Hk != 0 || d < 1 || n < 1) return -1;
    if (nthreads < 1) nthreads = 1;
    int64_t qoff = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int L = cu_seqlens[s + 1] - cu_seqlens[s];
        if (L < 0) return -1;
        if (L == 0) continue;
        const int ns = n < L ? n : L;
        double *Th = (double *)malloc(sizeof(double) * (size_t)Hq * (size_t)L);
        if (!Th) return -1;
        const int nt = nthreads < Hq ? nthreads : Hq;
        orc_head_job *jobs = (orc_head_job *)malloc(sizeof(orc_head_job) * (size_t)nt);
        pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
        for (int w = 0; w < nt; ++w) {
            jobs[w].q = q_last + (size_t)qoff * Hq * d;
            jobs[w].k = k + (size_t)cu_seqlens[s] * Hk * d;
            jobs[w].L = L; jobs[w].ns = ns; jobs[w].Hq = Hq; jobs[w].Hk = Hk; jobs[w].d = d;
            jobs[w].Th = Th; jobs[w].h_begin = w; jobs[w].h_step = nt;
        }
        if (nt == 1) {
            orc_head_worker(&jobs[0]);
        } else {
            for (int w = 0; w < nt; ++w) pthread_create(&tids[w], NULL, orc_head_worker, &jobs[w]);
            for (int w = 0; w < nt; ++w) pthread_join(tids[w], NULL);
        }
        const double denom = (double)ns * (double)Hq;
        for (int i = 0; i < L; ++i) {
            double acc = 0.0;
            for (int h = 0; h < Hq; ++h) acc += Th[(size_t)h * L + i];
            mass[cu_seqlens[s] + i] = acc / denom;
        }
        free(tids);
        free(jobs);
        free(Th);
        qoff += ns;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Block scores.  [UP] block-wise importance estimation: the sequence is cut  */
/* into fixed blocks of G tokens; block b of a sequence covers tokens         */
/* [bG, min((b+1)G, L)) and its score is the sum of their mass.  A shorter    */
/* last block keeps its own (smaller) sum.  cu_blocks is the exclusive prefix */
/* sum of nb_s = ceil(L_s / G).                                               */
/* ------------------------------------------------------------------------ */
int orc_block_scores(const double *mass, const int32_t *cu_seqlens, int num_seqs, int G,
                     double *scores, int32_t *cu_blocks)
{
    if (G < 1 || num_seqs < 0) return -1;
    cu_blocks[0] = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int L = cu_seqlens[s + 1] - cu_seqlens[s];
        const int nb = (L + G - 1) / G;
        for (int b = 0; b < nb; ++b) {
            const int end = (b + 1) * G < L ? (b + 1) * G : L;
            double acc = 0.0;
            for (int i = b * G; i < end; ++i) acc += mass[cu_seqlens[s] + i];
            scores[cu_blocks[s] + b] = acc;
        }
        cu_blocks[s + 1] = cu_blocks[s] + nb;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-p selection.  [UP] top-p selection: blocks are ordered by score        */
/* (highest first; equal scores by lower block index) and kept until the     */
/* cumulative score reaches p.  The crossing block is kept; p >= 1 keeps all; */
/* if rounding leaves the total short of p, every block is kept.             */
/* keep[] is in original block order; kept_tokens[s] counts the tokens of    */
/* the kept blocks.  cum_incl / cum_excl (nullable) receive, per block, the  */
/* fp64 cumulative mass at that block's rank, including / excluding it.      */
/* ------------------------------------------------------------------------ */
static const double *orc_sort_scores; /* comparator context; single-threaded */

static int orc_rank_cmp(const void *pa, const void *pb)
{
    const int a = *(const int *)pa, b = *(const int *)pb;
    const double sa = orc_sort_scores[a], sb = orc_sort_scores[b];
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return (a > b) - (a < b);
}

int orc_select_topp(const double *scores, const int32_t *cu_blocks, const int32_t *cu_seqlens,
                    int num_seqs, int G, double p, uint8_t *keep, int32_t *kept_tokens,
                    double *cum_incl, double *cum_excl)
{
    if (G < 1 || num_seqs < 0 || !(p > 0.0)) return -1;
    for (int s = 0; s < num_seqs; ++s) {
        const int nb = cu_blocks[s + 1] - cu_blocks[s];
        const int L = cu_seqlens[s + 1] - cu_seqlens[s];
        const double *sc = scores + cu_blocks[s];
        kept_tokens[s] = 0;
        if (nb == 0) continue;
        int *order = (int *)malloc(sizeof(int) * (size_t)nb);
        if (!order) return -1;
        for (int b = 0; b < nb; ++b) order[b] = b;
        orc_sort_scores = sc;
        qsort(order, (size_t)nb, sizeof(int), orc_rank_cmp);
        int last = nb - 1; /* rank of the last kept block */
        int found = 0;
        double c = 0.0;
        for (int r = 0; r < nb; ++r) {
            const double before = c;
            c += sc[order[r]];
            if (cum_incl) cum_incl[cu_blocks[s] + order[r]] = c;
            if (cum_excl) cum_excl[cu_blocks[s] + order[r]] = before;
            if (!found && p < 1.0 && c >= p) { last = r; found = 1; }
        }
        for (int b = 0; b < nb; ++b) keep[cu_blocks[s] + b] = 0;
        for (int r = 0; r <= last; ++r) {
            const int b = order[r];
            const int end = (b + 1) * G < L ? (b + 1) * G : L;
            keep[cu_blocks[s] + b] = 1;
            kept_tokens[s] += end - b * G;
        }
        free(order);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-k selection.  [UP] hyper-parameters paragraph: the ablation sets top-p  */
/* against keeping a fixed number of blocks per sequence (top-k).  Blocks are */
/* ranked exactly as for top-p (score descending, ties to the lower index)    */
/* and the first min(k, nb) ranks are kept.  Returns 0, or -1 on bad args.    */
/* ------------------------------------------------------------------------ */
int orc_select_topk(const double *scores, const int32_t *cu_blocks, const int32_t *cu_seqlens,
                    int num_seqs, int G, int k, uint8_t *keep, int32_t *kept_tokens)
{
    if (G < 1 || num_seqs < 0 || k < 1) return -1;
    for (int s = 0; s < num_seqs; ++s) {
        const int nb = cu_blocks[s + 1] - cu_blocks[s];
        const int L = cu_seqlens[s + 1] - cu_seqlens[s];
        const double *sc = scores + cu_blocks[s];
        kept_tokens[s] = 0;
        if (nb == 0) continue;
        int *order = (int *)malloc(sizeof(int) * (size_t)nb);
        if (!order) return -1;
        for (int b = 0; b < nb; ++b) order[b] = b;
        orc_sort_scores = sc;
        qsort(order, (size_t)nb, sizeof(int), orc_rank_cmp);
        for (int b = 0; b < nb; ++b) keep[cu_blocks[s] + b] = 0;
        for (int r = 0; r < nb && r < k; ++r) {
            const int b = order[r];
            const int end = (b + 1) * G < L ? (b + 1) * G : L;
            keep[cu_blocks[s] + b] = 1;
            kept_tokens[s] += end - b * G;
        }
        free(order);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Keep-last option.  [UP] system-integration paragraph: decode continues     */
/* from the end of each sequence.  As an option applied after either          */
/* selection, the last block of every non-empty sequence (its most recent     */
/* tokens) is also kept and kept_tokens counts it; the method as the pages    */
/* state it leaves this off.  Returns 0, or -1 on bad args.                   */
/* ------------------------------------------------------------------------ */
int orc_keep_last_block(const int32_t *cu_blocks, const int32_t *cu_seqlens, int num_seqs,
                        int G, uint8_t *keep, int32_t *kept_tokens)
{
    if (G < 1 || num_seqs < 0) return -1;
    for (int s = 0; s < num_seqs; ++s) {
        const int nb = cu_blocks[s + 1] - cu_blocks[s];
        const int L = cu_seqlens[s + 1] - cu_seqlens[s];
        if (nb == 0) continue;
        const int b = nb - 1;
        if (!keep[cu_blocks[s] + b]) {
            keep[cu_blocks[s] + b] = 1;
            kept_tokens[s] += L - b * G;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Compaction.  [UP] sparsity propagation: every later sub-layer sees only    */
/* the kept tokens; [UP] system integration: the positions of kept tokens    */
/* travel with them so decode can address the KV cache.  For each sequence   */
/* in order and each kept block in ascending order, the block's rows of x    */
/* and pos are appended; src_idx (nullable) records each output row's        */
/* source row; cu_out is the compacted batch's cu_seqlens.  x_out / pos_out  */
/* may be NULL to skip that copy.  Returns the number of kept rows, or -1.   */
/* ------------------------------------------------------------------------ */
int64_t orc_compact(const uint16_t *x, const int32_t *pos, int64_t hidden,
                    const int32_t *cu_seqlens, int num_seqs, int G, const uint8_t *keep,
                    const int32_t *cu_blocks, uint16_t *x_out, int32_t *pos_out,
                    int32_t *cu_out, int32_t *src_idx)
{
    if (G < 1 || num_seqs < 0 || hidden < 0) return -1;
    int64_t o = 0;
    cu_out[0] = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int L = cu_seqlens[s + 1] - cu_seqlens[s];
        const int nb = cu_blocks[s + 1] - cu_blocks[s];
        for (int b = 0; b < nb; ++b) {
            if (!keep[cu_blocks[s] + b]) continue;
            const int end = (b + 1) * G < L ? (b + 1) * G : L;
            for (int i = b * G; i < end; ++i) {
                const int64_t src = (int64_t)cu_seqlens[s] + i;
                if (x_out)
                    memcpy(x_out + o * hidden, x + src * hidden, sizeof(uint16_t) * (size_t)hidden);
                if (pos_out) pos_out[o] = pos[src];
                if (src_idx) src_idx[o] = (int32_t)src;
                ++o;
            }
        }
        cu_out[s + 1] = (int32_t)o;
    }
    return o;
}

/* Kept blocks as a block-CSR matrix (FlashPrefill V2 review, key-terms
 * section: the active blocks handed to a sparse-attention kernel as a CSR
 * index).  The plain definition: for each sequence in order, the numbers
 * (0-based within the sequence) of its kept blocks, ascending; indptr[s] =
 * kept blocks of the sequences before s.  Returns the number of kept blocks,
 * or -1 for bad arguments. */
int64_t orc_block_csr(const uint8_t *keep, const int32_t *cu_blocks, int B, int32_t *indptr,
                      int32_t *indices) {
    if (B < 0 || !cu_blocks || !indptr) return -1;
    int64_t nnz = 0;
    for (int s = 0; s < B; ++s) {
        indptr[s] = (int32_t)nnz;
        for (int32_t b = cu_blocks[s]; b < cu_blocks[s + 1]; ++b)
            if (keep[b]) indices[nnz++] = b - cu_blocks[s];
    }
    indptr[B] = (int32_t)nnz;
    return nnz;
}
