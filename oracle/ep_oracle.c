/*
 * CPU oracle for the MoE expert-parallel dispatch/combine hot path:
 * layout counting, notify prefix sums, channelised dispatch and fp32 combine.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package
 * smoke check and the benchmark's CPU-baseline leg load this library.  It is
 * a plain, slow, single-threaded restatement of the definitions, written so a
 * reader can check it against the pages by eye.  It shares no code, header or
 * table with the CUDA path.
 *
 * Pages (cited by title and section):
 *   [IN]  "notify_dispatch (internode.cu)" notes on DeepEP - sm0 stages 3-6,
 *         sm1..x stages 1-3 (per-channel counting and prefix sums).
 *   [CH]  "cuda】deepep" - channels as a spatial partition of a rank's tokens.
 *   [RT]  mscclpp src/ext/ep/ht_runtime.cc - MoEHighThroughputRuntime::
 *         getDispatchLayout / intranodeNotifyDispatch / internodeNotifyDispatch /
 *         intranodeDispatch / internodeDispatch / intranodeCombine.
 *   [AR]  "CUDA与DeepEP：分布式MoE系统中的高效通信机制解析" - 2.2 rank-to-node
 *         mapping, 3.2 two-level reduction, 4.1 SrcInfo, 4.2 combine routing.
 *
 * Notation: R ranks, N = max(1, R/8) nodes (node of rank r is r/8), T tokens
 * per rank, K top-k slots, E experts, E_loc = E/R experts per rank, H hidden
 * size (bf16 elements), C channels.  Every rank-indexed array is stacked:
 * x[R][T][H], topk_idx[R][T][K] and so on, all contiguous in C order.
 *
 * Readings where the pages leave a step open:
 *   P1 channel c of a rank covers tokens [min(c*q,T), min((c+1)*q,T)), q=ceil(T/C)
 *   P2 the node-level receive prefix of rank r sums, over source nodes m, what
 *      rank m*8 + r%8 sends to node r/8
 *   P3 recv_channel_offset[r][s][c] is the first row of block (s,c) inside r's
 *      receive region
 *   P4 src_info is the pair (source rank, source token)
 *   P5 received top-k ids are re-expressed as local expert ids (or -1), and a
 *      weight is kept only where its expert lives on the receiving rank
 *   P6 combine is an unweighted fp32 sum over contributing ranks in ascending
 *      rank order, rounded once to bf16 (round to nearest even)
 *   P7 per-expert counts count every slot, a token counts once per rank
 */
#include <stddef.h>
#include <stdint.h>
#include <math.h>
#include <string.h>

#define NODE_SIZE 8 /* ranks per node: NUM_MAX_NVL_PEERS, [AR] 2.2 */

/* Planted mistakes.  The default build (ORACLE_MUTANT 0) has none.  The
 * tests compile copies with ORACLE_MUTANT = 1..11, each carrying one plausible
 * error, and check that the pins reject every one of them. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUT(n) (ORACLE_MUTANT == (n))

static int nodes_of(int R) { return R <= NODE_SIZE ? 1 : R / NODE_SIZE; }

int oracle_num_nodes(int R) { return nodes_of(R); }

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32.  bf16 is the upper half of an IEEE binary32 word.  Rounding
 * to nearest, ties to even: add half of the dropped range, plus one when the
 * kept part is odd, then truncate.  NaN stays NaN (quiet bit set). */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_odd = (u >> 16) & 1u;
    if (!MUT(8)) u += 0x7fffu + keep_odd;
    return (uint16_t)(u >> 16);
}

/* Exposed so the tests can pin the rounding against an independent library. */
void oracle_f32_to_bf16(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Channel token range, reading P1 ([CH]: a channel is a contiguous lane of a
 * rank's tokens; [RT] uses num_channels = num_sms / 2). */
static void channel_range(int T, int C, int c, int* begin, int* end)
{
    int q = MUT(1) ? T / C : (T + C - 1) / C;
    if (q == 0) q = 1;
    int64_t b = (int64_t)c * q, e = (int64_t)(c + 1) * q;
    *begin = (int)(b < T ? b : T);
    *end = (int)(e < T ? e : T);
}

/* ------------------------------------------------------------------------ */
/* Step 1: layout counting.  [RT] getDispatchLayout: from topk_idx produce
 * num_tokens_per_rank, num_tokens_per_rdma_rank, num_tokens_per_expert and
 * is_token_in_rank; [IN] sm0 stage 3 shows the same three count vectors being
 * packed per destination node.  An expert e >= 0 lives on rank e / E_loc
 * ([RT] num_local_experts = numExperts / num_ranks); -1 marks an empty slot.
 * Returns 0, or -1 when an id is outside [-1, E). */
int oracle_layout(int R, int T, int K, int E,
                  const int64_t* topk_idx,          /* [R][T][K] */
                  int32_t* num_tokens_per_rank,     /* [R][R]    */
                  int32_t* num_tokens_per_rdma_rank,/* [R][N]    */
                  int32_t* num_tokens_per_expert,   /* [R][E]    */
                  uint8_t* is_token_in_rank)        /* [R][T][R] */
{
    const int N = nodes_of(R);
    const int E_loc = E / R;
    memset(num_tokens_per_rank, 0, sizeof(int32_t) * (size_t)R * R);
    memset(num_tokens_per_rdma_rank, 0, sizeof(int32_t) * (size_t)R * N);
    memset(num_tokens_per_expert, 0, sizeof(int32_t) * (size_t)R * E);
    for (int s = 0; s < R; ++s) {
        for (int t = 0; t < T; ++t) {
            uint8_t* in_rank = is_token_in_rank + ((size_t)s * T + t) * R;
            memset(in_rank, 0, (size_t)R);
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[((size_t)s * T + t) * K + k];
                if (e < -1 || e >= E) return -1;
                if (e < 0) continue;
                num_tokens_per_expert[(size_t)s * E + e] += 1; /* P7: every slot */
                in_rank[e / E_loc] = MUT(7) ? (uint8_t)(in_rank[e / E_loc] + 1) : 1;
            }
            for (int r = 0; r < R; ++r) num_tokens_per_rank[(size_t)s * R + r] += in_rank[r];
            for (int n = 0; n < N; ++n) {
                int any = 0;
                for (int r = n * NODE_SIZE; r < R && r < (n + 1) * NODE_SIZE; ++r) any |= in_rank[r];
                num_tokens_per_rdma_rank[(size_t)s * N + n] += any;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: notify prefix sums.  Follows [IN]:
 *   sm1..x stages 1-3: per channel, count the tokens sent to each rank and to
 *     each node, then prefix over channels -> gbl_channel_prefix_matrix and
 *     rdma_channel_prefix_matrix (inclusive);
 *   sm0 stage 6: prefix of per-rank counts over global source rank ->
 *     recv_gbl_rank_prefix_sum (ordering by source rank), total -> the receive
 *     counter; prefix over source nodes -> recv_rdma_rank_prefix_sum (P2);
 *     per-expert sum rounded up to expert_alignment.
 * [RT] intranodeNotifyDispatch names the same result rank_prefix_matrix,
 * shaped [num_ranks, num_ranks] (source-major), and channel_prefix_matrix.
 * The single receive pool (recv_base) and the row map send_pos are this
 * library's own layout: all destination regions sit back to back in one pool,
 * and send_pos[s][t][r] is the row of token (s,t) inside rank r's region (the
 * role of [RT]'s send_head), or -1. */
int oracle_notify(int R, int T, int E, int C, int expert_alignment,
                  const uint8_t* is_token_in_rank,         /* [R][T][R] */
                  const int32_t* num_tokens_per_rank,      /* [R][R]    */
                  const int32_t* num_tokens_per_rdma_rank, /* [R][N]    */
                  const int32_t* num_tokens_per_expert,    /* [R][E]    */
                  int32_t* rank_prefix_matrix,             /* [R src][R dst]  */
                  int32_t* gbl_channel_prefix_matrix,      /* [R src][R dst][C] */
                  int32_t* rdma_channel_prefix_matrix,     /* [R src][N][C]  */
                  int32_t* recv_gbl_rank_prefix_sum,       /* [R dst][R src] */
                  int32_t* recv_rdma_rank_prefix_sum,      /* [R dst][N]     */
                  int32_t* recv_channel_offset,            /* [R dst][R src][C] */
                  int32_t* num_recv_tokens,                /* [R] */
                  int32_t* num_rdma_recv_tokens,           /* [R] */
                  int32_t* num_recv_tokens_per_expert,     /* [R][E_loc] */
                  int64_t* recv_base,                      /* [R+1] */
                  int32_t* send_pos)                       /* [R src][T][R dst] */
{
    const int N = nodes_of(R);
    const int E_loc = E / R;
    if (C < 1 || expert_alignment < 1) return -1;

    /* [IN] sm1..x: per-channel counts and their inclusive prefix over channels */
    for (int s = 0; s < R; ++s) {
        for (int r = 0; r < R; ++r) {
            int32_t run = 0;
            for (int c = 0; c < C; ++c) {
                int b, e;
                channel_range(T, C, c, &b, &e);
                for (int t = b; t < e; ++t) run += is_token_in_rank[((size_t)s * T + t) * R + r];
                gbl_channel_prefix_matrix[((size_t)s * R + r) * C + c] = run;
            }
        }
        for (int n = 0; n < N; ++n) {
            int32_t run = 0;
            for (int c = 0; c < C; ++c) {
                int b, e;
                channel_range(T, C, c, &b, &e);
                for (int t = b; t < e; ++t) {
                    int any = 0;
                    for (int r = n * NODE_SIZE; r < R && r < (n + 1) * NODE_SIZE; ++r)
                        any |= is_token_in_rank[((size_t)s * T + t) * R + r];
                    run += any;
                }
                rdma_channel_prefix_matrix[((size_t)s * N + n) * C + c] = run;
            }
        }
    }

    /* [IN] sm0 stage 6: prefix over global source rank i = rdma*8 + nvl */
    for (int r = 0; r < R; ++r) {
        int32_t run = 0;
        for (int s = 0; s < R; ++s) {
            run += num_tokens_per_rank[(size_t)s * R + r];
            rank_prefix_matrix[(size_t)s * R + r] = run;
            recv_gbl_rank_prefix_sum[(size_t)r * R + s] = run;
        }
        num_recv_tokens[r] = run;
    }

    /* [IN] sm0 stage 6, reading P2: rank r receives for its node from the
     * same-GPU-index peer of every node m */
    for (int r = 0; r < R; ++r) {
        int32_t run = 0;
        for (int m = 0; m < N; ++m) {
            int peer = MUT(4) ? m * NODE_SIZE + r / NODE_SIZE : m * NODE_SIZE + r % NODE_SIZE;
            run += num_tokens_per_rdma_rank[(size_t)peer * N + r / NODE_SIZE];
            recv_rdma_rank_prefix_sum[(size_t)r * N + m] = run;
        }
        num_rdma_recv_tokens[r] = run;
    }

    /* [IN] sm0 stage 6: per-expert receive counts, rounded up to the alignment */
    for (int r = 0; r < R; ++r) {
        for (int j = 0; j < E_loc; ++j) {
            int64_t sum = 0;
            for (int s = 0; s < R; ++s) sum += num_tokens_per_expert[(size_t)s * E + r * E_loc + j];
            sum = MUT(5) ? sum / expert_alignment * expert_alignment
                         : (sum + expert_alignment - 1) / expert_alignment * expert_alignment;
            num_recv_tokens_per_expert[(size_t)r * E_loc + j] = (int32_t)sum;
        }
    }

    /* single pool: destination regions back to back, ascending rank */
    recv_base[0] = 0;
    for (int r = 0; r < R; ++r) recv_base[r + 1] = recv_base[r] + num_recv_tokens[r];

    /* P3: first row of block (s,c) in r's region = tokens of earlier source
     * ranks plus tokens of earlier channels of the same source rank */
    for (int r = 0; r < R; ++r)
        for (int s = 0; s < R; ++s)
            for (int c = 0; c < C; ++c) {
                int32_t before_s = s > 0 ? rank_prefix_matrix[(size_t)(s - (MUT(2) ? 0 : 1)) * R + r] : 0;
                int32_t before_c = c > 0 ? gbl_channel_prefix_matrix[((size_t)s * R + r) * C + c - 1] : 0;
                recv_channel_offset[((size_t)r * R + s) * C + c] = before_s + before_c;
            }

    /* Row of each (s,t,r): block offset plus the running index inside the
     * channel, visiting tokens in (source rank, channel, token) order. */
    for (int s = 0; s < R; ++s)
        for (int c = 0; c < C; ++c) {
            int b, e;
            channel_range(T, C, c, &b, &e);
            for (int r = 0; r < R; ++r) {
                int32_t i = 0;
                for (int t = b; t < e; ++t) {
                    size_t at = ((size_t)s * T + t) * R + r;
                    send_pos[at] = is_token_in_rank[at]
                                       ? recv_channel_offset[((size_t)r * R + s) * C + c] + i++
                                       : -1;
                }
            }
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 3: dispatch of one source token (s,t) to every rank it is routed to.
 * [RT] intranodeDispatch / internodeDispatch: the receive side holds recv_x,
 * recv_topk_idx (int64), recv_topk_weights (fp32) and the source index / meta;
 * [AR] 4.1 gives src_info as {src_rank, src_idx} (P4).  Readings P5 for the
 * top-k fields.  Rows land at recv_base[r] + send_pos[s][t][r]. */
static int dispatch_token(int R, int T, int K, int E, size_t row_bytes, int s, int t,
                          const void* x_row, const float* scales_row, int S,
                          const int64_t* topk_idx, const float* topk_w,
                          const int32_t* send_pos, const int64_t* recv_base,
                          void* recv_x, float* recv_x_scales, int64_t* recv_topk_idx,
                          float* recv_topk_w, int32_t* recv_src_info)
{
    const int E_loc = E / R;
    for (int r = 0; r < R; ++r) {
        int32_t pos = send_pos[((size_t)s * T + t) * R + r];
        if (pos < 0) continue;
        int64_t row = recv_base[r] + pos;
        if (row >= recv_base[r + 1]) return -1; /* row outside r's region */
        if (recv_x && x_row) memcpy((uint8_t*)recv_x + (size_t)row * row_bytes, x_row, row_bytes);
        if (recv_x_scales && scales_row)
            memcpy(recv_x_scales + (size_t)row * S, scales_row, sizeof(float) * (size_t)S);
        for (int k = 0; recv_topk_idx && k < K; ++k) { /* cached mode: no top-k */
            int64_t e = topk_idx[((size_t)s * T + t) * K + k];
            int here = e >= 0 && e / E_loc == r;
            recv_topk_idx[(size_t)row * K + k] = here ? e - (MUT(6) ? 0 : (int64_t)r * E_loc) : -1;
            recv_topk_w[(size_t)row * K + k] = here ? topk_w[((size_t)s * T + t) * K + k] : 0.0f;
        }
        if (recv_src_info) {
            recv_src_info[(size_t)row * 2 + 0] = s;
            recv_src_info[(size_t)row * 2 + 1] = t;
        }
    }
    return 0;
}

/* Whole dispatch in the pages' order: source rank, channel, token.  x and
 * recv_x may both be NULL to produce only the metadata (for shapes whose
 * payload does not fit in host memory).  In cached mode ([RT]
 * intranodeDispatch with cachedMode, num_experts 0) the top-k is not
 * dispatched: recv_topk_idx / recv_topk_w are NULL, and recv_src_info may be
 * NULL as well.  Returns -1 when a row falls outside its destination's
 * region. */
int oracle_dispatch(int R, int T, int K, int E, int H, int C,
                    const uint16_t* x,        /* [R][T][H] or NULL */
                    const int64_t* topk_idx,  /* [R][T][K] */
                    const float* topk_w,      /* [R][T][K] */
                    const int32_t* send_pos,  /* [R][T][R] */
                    const int64_t* recv_base, /* [R+1] */
                    uint16_t* recv_x,         /* [rows][H] or NULL */
                    int64_t* recv_topk_idx,   /* [rows][K] */
                    float* recv_topk_w,       /* [rows][K] */
                    int32_t* recv_src_info)   /* [rows][2] */
{
    for (int s = 0; s < R; ++s)
        for (int c = 0; c < C; ++c) {
            int b, e;
            channel_range(T, C, c, &b, &e);
            for (int t = b; t < e; ++t)
                if (dispatch_token(R, T, K, E, sizeof(uint16_t) * (size_t)H, s, t,
                                   x ? x + ((size_t)s * T + t) * H : NULL, NULL, 0, topk_idx, topk_w,
                                   send_pos, recv_base, recv_x, NULL, recv_topk_idx, recv_topk_w,
                                   recv_src_info) != 0)
                    return -1;
        }
    return 0;
}

/* FP8 dispatch: [RT] intranodeDispatch / internodeDispatch with an element
 * size of one byte and num_scales fp32 scales per token (x_scales ->
 * recv_x_scales).  The same placement as oracle_dispatch; each row is H bytes
 * and its scales row travels with it.  x_scales / recv_x_scales may be NULL
 * when S == 0, the top-k arrays NULL in cached mode. */
int oracle_dispatch_fp8(int R, int T, int K, int E, int H, int C, int S,
                        const uint8_t* x,          /* [R][T][H] */
                        const float* x_scales,     /* [R][T][S] or NULL */
                        const int64_t* topk_idx,   /* [R][T][K] or NULL */
                        const float* topk_w,       /* [R][T][K] or NULL */
                        const int32_t* send_pos,   /* [R][T][R] */
                        const int64_t* recv_base,  /* [R+1] */
                        uint8_t* recv_x,           /* [rows][H] */
                        float* recv_x_scales,      /* [rows][S] or NULL */
                        int64_t* recv_topk_idx,    /* [rows][K] or NULL */
                        float* recv_topk_w,        /* [rows][K] or NULL */
                        int32_t* recv_src_info)    /* [rows][2] or NULL */
{
    for (int s = 0; s < R; ++s)
        for (int c = 0; c < C; ++c) {
            int b, e;
            channel_range(T, C, c, &b, &e);
            for (int t = b; t < e; ++t)
                if (dispatch_token(R, T, K, E, (size_t)H, s, t, x + ((size_t)s * T + t) * H,
                                   x_scales ? x_scales + ((size_t)s * T + t) * S : NULL, S, topk_idx,
                                   topk_w, send_pos, recv_base, recv_x, recv_x_scales, recv_topk_idx,
                                   recv_topk_w, recv_src_info) != 0)
                    return -1;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 4: combine, reading P6.  [RT] intranodeCombine reduces every token's
 * contributions from all ranks into combined_x (bf16) and combined_topk_weights;
 * [AR] 4.2 routes each received row back to (src_rank, src_idx).  The rows of
 * token (s,t) are found through send_pos, summed in fp32 in ascending rank
 * order starting from +0, and rounded once.  A token with no destination
 * combines to zero.  y_w / combined_w may be NULL.  Returns -1 when a row
 * lies outside y. */
int oracle_combine(int R, int T, int K, int H, int64_t y_rows,
                   const uint16_t* y,        /* [y_rows][H] */
                   const float* y_w,         /* [rows][K] or NULL */
                   const int32_t* send_pos,  /* [R][T][R] */
                   const int64_t* recv_base, /* [R+1] */
                   uint16_t* combined_x,     /* [R][T][H] */
                   float* combined_w)        /* [R][T][K] or NULL */
{
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t) {
            const int32_t* pos = send_pos + ((size_t)s * T + t) * R;
            for (int r = 0; r < R; ++r)
                if (pos[r] >= 0 && (recv_base[r] + pos[r] >= y_rows || recv_base[r] + pos[r] < 0))
                    return -1;
            uint16_t* out = combined_x + ((size_t)s * T + t) * H;
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int i = 0; i < R; ++i) {
                    int r = MUT(3) ? R - 1 - i : i;
                    if (pos[r] >= 0) acc += bf16_to_f32(y[(size_t)(recv_base[r] + pos[r]) * H + h]);
                }
                out[h] = f32_to_bf16(acc);
            }
            if (y_w && combined_w) {
                for (int k = 0; k < K; ++k) {
                    float acc = 0.0f;
                    for (int i = 0; i < R; ++i) {
                        int r = MUT(11) ? R - 1 - i : i;
                        if (pos[r] >= 0) acc += y_w[(size_t)(recv_base[r] + pos[r]) * K + k];
                    }
                    combined_w[((size_t)s * T + t) * K + k] = acc;
                }
            }
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Low-latency (per-expert packed) layout.  The pages give only this mode's
 * transport ([RT] "Intra-node LL fast path setup": peer pointers, fabric IPC,
 * proxy threads for LL combine); the plain reading used here:
 *   - every non-masked top-k slot (s,t,k) that names expert e is one row of
 *     e's receive buffer (a token travels once per expert, not per rank);
 *   - rows of a buffer are in ascending (source rank, token, slot) order;
 *   - layout_range[e][s] = (first row, rows) of source s in e's buffer, and
 *     count[e] = rows in e's buffer;
 *   - LL combine applies the routing weights: out[s][t] =
 *     bf16_rne(sum over valid k ascending of fma(w[s][t][k], y[e_k][row_k], acc))
 *     starting from +0, with the fused multiply-add rounded once per step.
 * Buffers hold `cap` rows each; a slot whose row would reach cap is dropped
 * (pos -1).  Returns -1 on an expert id outside [-1, E), 1 when a row was
 * dropped, else 0. */
int oracle_ll_layout(int R, int T, int K, int E, int cap,
                     const int64_t* topk_idx,  /* [R][T][K] */
                     int32_t* slot_pos,        /* [R][T][K] row inside its expert's buffer, or -1 */
                     int32_t* layout_range,    /* [E][R][2] */
                     int32_t* count)           /* [E] */
{
    int dropped = 0;
    memset(count, 0, sizeof(int32_t) * (size_t)E);
    for (int s = 0; s < R; ++s) {
        for (int e = 0; e < E; ++e) {
            layout_range[((size_t)e * R + s) * 2 + 0] = count[e];
            layout_range[((size_t)e * R + s) * 2 + 1] = 0;
        }
        for (int t = 0; t < T; ++t)
            for (int kk = 0; kk < K; ++kk) {
                int k = MUT(10) ? K - 1 - kk : kk;
                size_t at = ((size_t)s * T + t) * K + k;
                int64_t e = topk_idx[at];
                if (e < -1 || e >= E) return -1;
                if (e < 0) {
                    slot_pos[at] = -1;
                    continue;
                }
                int32_t row = count[e];
                count[e] += 1;
                layout_range[((size_t)e * R + s) * 2 + 1] += 1;
                if (row >= cap) {
                    slot_pos[at] = -1;
                    dropped = 1;
                } else {
                    slot_pos[at] = row;
                }
            }
    }
    return dropped;
}

/* LL dispatch: copy each token row to every (expert, row) its slots name. */
int oracle_ll_dispatch(int R, int T, int K, int E, int H, int cap,
                       const uint16_t* x,          /* [R][T][H] */
                       const int64_t* topk_idx,    /* [R][T][K] */
                       const int32_t* slot_pos,    /* [R][T][K] */
                       uint16_t* recv_x,           /* [E][cap][H] */
                       int32_t* recv_src_info)     /* [E][cap][2] */
{
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t)
            for (int k = 0; k < K; ++k) {
                size_t at = ((size_t)s * T + t) * K + k;
                int64_t e = topk_idx[at];
                int32_t row = slot_pos[at];
                if (e < 0 || row < 0) continue;
                if (row >= cap || e >= E) return -1;
                size_t dst = (size_t)e * cap + row;
                memcpy(recv_x + dst * H, x + ((size_t)s * T + t) * H, sizeof(uint16_t) * (size_t)H);
                recv_src_info[dst * 2 + 0] = s;
                recv_src_info[dst * 2 + 1] = t;
            }
    return 0;
}

/* LL combine: weighted sum over the token's slots, ascending k. */
int oracle_ll_combine(int R, int T, int K, int E, int H, int cap,
                      const uint16_t* y,          /* [E][cap][H] */
                      const int64_t* topk_idx,    /* [R][T][K] */
                      const float* topk_w,        /* [R][T][K] */
                      const int32_t* slot_pos,    /* [R][T][K] */
                      uint16_t* combined_x)       /* [R][T][H] */
{
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t) {
            size_t tok = (size_t)s * T + t;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[tok * K + k];
                int32_t row = slot_pos[tok * K + k];
                if (e >= E || row >= cap) return -1;
            }
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int k = 0; k < K; ++k) {
                    int64_t e = topk_idx[tok * K + k];
                    int32_t row = slot_pos[tok * K + k];
                    if (e < 0 || row < 0) continue;
                    if (MUT(9)) {
                        float prod = topk_w[tok * K + k] * bf16_to_f32(y[((size_t)e * cap + row) * H + h]);
                        acc += prod;
                    } else {
                        acc = fmaf(topk_w[tok * K + k], bf16_to_f32(y[((size_t)e * cap + row) * H + h]), acc);
                    }
                }
                combined_x[tok * H + h] = f32_to_bf16(acc);
            }
        }
    return 0;
}
