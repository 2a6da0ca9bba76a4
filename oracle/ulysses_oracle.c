/*
 * CPU oracle for the two DeepSpeed-Ulysses layout changes -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load this file's
 * library. It shares no code, header or constant with the CUDA path.
 *
 * Layouts (B batch, L sequence, H heads, d per-head width, P shards, Lp = L/P, Hp = H/P):
 *   token-sharded  X[r][b][t][h][e]   shard r owns global tokens s = r*Lp + t, all H heads
 *   head-sharded   Y[g][b][s][j][e]   group g owns heads h = g*Hp + j, all L tokens
 *
 * seq->head is the first all-to-all of the paper (summary page, section 3.4.1 "The
 * layout transformation: sequence-partitioned to head-partitioned"; pinyu.ai page,
 * "Use the other independent axis"): every sender cuts its heads into P contiguous
 * groups, and receiver g takes group g from every sender and joins the token blocks
 * along the sequence in sender order. head->seq is the second all-to-all ("After
 * attention: the reverse transformation"), the inverse permutation.
 *
 * Elements are moved as opaque bytes (elem_bytes wide), so bf16 bit patterns -- NaN
 * payloads and denormals included -- and fp64 values both pass through unchanged.
 *
 * Return value: 0 on success, 1 if the shape is invalid (P, H or L not positive, H or L
 * not divisible by P, elem_bytes not in {1, 2, 4, 8}).
 */
#include <stdint.h>
#include <string.h>

static int shape_ok(int64_t P, int64_t B, int64_t L, int64_t H, int64_t d, int64_t eb)
{
    if (P <= 0 || B < 0 || L < 0 || H <= 0 || d <= 0) return 0;
    if (L % P != 0 || H % P != 0) return 0;
    if (eb != 1 && eb != 2 && eb != 4 && eb != 8) return 0;
    return 1;
}

static void move_one(char *dst, const char *src, int64_t eb)
{
    memcpy(dst, src, (size_t)eb);
}

/* Y[g][b][s][j][e] = X[s / Lp][b][s % Lp][g*Hp + j][e]; loops run over the source. */
int oracle_seq_to_head(int64_t P, int64_t B, int64_t L, int64_t H, int64_t d, int64_t elem_bytes,
                       const void *x, void *y)
{
    if (!shape_ok(P, B, L, H, d, elem_bytes)) return 1;
    const int64_t Lp = L / P, Hp = H / P;
    const char *X = (const char *)x;
    char *Y = (char *)y;
    for (int64_t r = 0; r < P; ++r)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t t = 0; t < Lp; ++t)
                for (int64_t h = 0; h < H; ++h)
                    for (int64_t e = 0; e < d; ++e) {
                        const int64_t s = r * Lp + t;      /* global token index  */
                        const int64_t g = h / Hp;          /* receiving group     */
                        const int64_t j = h % Hp;          /* head within group   */
                        const int64_t src = (((r * B + b) * Lp + t) * H + h) * d + e;
                        const int64_t dst = (((g * B + b) * L + s) * Hp + j) * d + e;
                        move_one(Y + dst * elem_bytes, X + src * elem_bytes, elem_bytes);
                    }
    return 0;
}

/* Z[r][b][t][h][e] = Y[h / Hp][b][r*Lp + t][h % Hp][e]; loops run over the destination. */
int oracle_head_to_seq(int64_t P, int64_t B, int64_t L, int64_t H, int64_t d, int64_t elem_bytes,
                       const void *y, void *z)
{
    if (!shape_ok(P, B, L, H, d, elem_bytes)) return 1;
    const int64_t Lp = L / P, Hp = H / P;
    const char *Y = (const char *)y;
    char *Z = (char *)z;
    for (int64_t r = 0; r < P; ++r)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t t = 0; t < Lp; ++t)
                for (int64_t h = 0; h < H; ++h)
                    for (int64_t e = 0; e < d; ++e) {
                        const int64_t dst = (((r * B + b) * Lp + t) * H + h) * d + e;
                        const int64_t src = (((h / Hp * B + b) * L + r * Lp + t) * Hp + h % Hp) * d + e;
                        move_one(Z + dst * elem_bytes, Y + src * elem_bytes, elem_bytes);
                    }
    return 0;
}

/* bf16 bit pattern -> fp64, exactly: a bf16 value is the top half of an IEEE fp32. */
void oracle_bf16_to_f64(int64_t n, const uint16_t *in, double *out)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t w = (uint32_t)in[i] << 16;
        float f;
        memcpy(&f, &w, sizeof f);
        out[i] = (double)f;
    }
}

/*
 * Grouped K/V heads (GQA/MQA): K and V carry Hkv heads shared by groups of H/Hkv query heads
 * (paper summary section 6, "Architecture generalization to grouped-query and multi-query
 * attention"; pinyu.ai page, "Head-count constraints"). Two regimes:
 *   Hkv % P == 0: receiver g gets the contiguous K/V heads [g*Hkv/P, (g+1)*Hkv/P), just as for Q;
 *   P % Hkv == 0: every receiver gets one K/V head, head g / (P/Hkv): each head is replicated
 *                 on P/Hkv receivers (the replication the pinyu.ai page mentions).
 * Head-sharded K/V: [P][B][L][Hkvp][d] with Hkvp = Hkv/P or 1.
 * Returns 1 for shapes outside both regimes.
 */
static int kv_shape(int64_t P, int64_t Hkv, int64_t *Hkvp, int64_t *rep)
{
    if (P <= 0 || Hkv <= 0) return 0;
    if (Hkv % P == 0) { *Hkvp = Hkv / P; *rep = 1; return 1; }
    if (P % Hkv == 0) { *Hkvp = 1; *rep = P / Hkv; return 1; }
    return 0;
}

/* source K/V head of slot j on receiver g */
static int64_t kv_source_head(int64_t g, int64_t j, int64_t Hkvp, int64_t rep)
{
    return rep == 1 ? g * Hkvp + j : g / rep;
}

/* Y[g][b][s][j][e] = X[s / Lp][b][s % Lp][kv_source_head(g, j)][e]; loops over the destination. */
int oracle_kv_seq_to_head(int64_t P, int64_t B, int64_t L, int64_t Hkv, int64_t d, int64_t elem_bytes,
                          const void *x, void *y)
{
    int64_t Hkvp, rep;
    if (!kv_shape(P, Hkv, &Hkvp, &rep) || !shape_ok(P, B, L, P, d, elem_bytes)) return 1;
    const int64_t Lp = L / P;
    const char *X = (const char *)x;
    char *Y = (char *)y;
    for (int64_t g = 0; g < P; ++g)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t s = 0; s < L; ++s)
                for (int64_t j = 0; j < Hkvp; ++j)
                    for (int64_t e = 0; e < d; ++e) {
                        const int64_t hs = kv_source_head(g, j, Hkvp, rep);
                        const int64_t src = (((s / Lp * B + b) * Lp + s % Lp) * Hkv + hs) * d + e;
                        const int64_t dst = (((g * B + b) * L + s) * Hkvp + j) * d + e;
                        move_one(Y + dst * elem_bytes, X + src * elem_bytes, elem_bytes);
                    }
    return 0;
}

/* The adjoint of oracle_kv_seq_to_head on fp64 values (used for dK, dV):
 *   Z[r][b][t][h][e] = sum over (g, j) with kv_source_head(g, j) == h of Y[g][b][r*Lp + t][j][e].
 * Without replication every head has exactly one source and this is the inverse permutation. */
int oracle_kv_head_to_seq_sum(int64_t P, int64_t B, int64_t L, int64_t Hkv, int64_t d, const double *y, double *z)
{
    int64_t Hkvp, rep;
    if (!kv_shape(P, Hkv, &Hkvp, &rep) || L % P != 0 || B < 0 || d <= 0) return 1;
    const int64_t Lp = L / P;
    for (int64_t i = 0; i < P * B * Lp * Hkv * d; ++i) z[i] = 0.0;
    for (int64_t g = 0; g < P; ++g)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t s = 0; s < L; ++s)
                for (int64_t j = 0; j < Hkvp; ++j)
                    for (int64_t e = 0; e < d; ++e) {
                        const int64_t hs = kv_source_head(g, j, Hkvp, rep);
                        const int64_t dst = (((s / Lp * B + b) * Lp + s % Lp) * Hkv + hs) * d + e;
                        z[dst] += y[(((g * B + b) * L + s) * Hkvp + j) * d + e];
                    }
    return 0;
}
