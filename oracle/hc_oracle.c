/*
 * hc_oracle.c -- plain, slow CPU oracle for the HCCL-style AllReduce /
 * ReduceScatter / AllGather schedules (Ring, Recursive Halving-Doubling,
 * hierarchical Pipeline).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links
 * or calls this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA path: its segment layout, loop slicer, schedule
 * generators and arithmetic are written here a second time, from the pages.
 *
 * What it computes (sources are the pages' titles and sections):
 *  - Definition: "AllReduce的数学抽象与问题定义" (HCCL Ring vs RHD article):
 *    Y[j] = (+)_i X_i[j] on every rank; ReduceScatter gives rank r segment r
 *    of Y; AllGather gives every rank the concatenation of the segments.
 *  - Ring: "Ring AllReduce带宽最优的环形流水线" (same article) and the
 *    "AllReduce算法实现" section of the HCCL topology / AllReduce article:
 *    P-1 reduce steps around the ring, then P-1 copy steps.
 *  - RHD: "Recursive Halving-Doubling短消息场景的延迟优势" (first article),
 *    "算法描述" and Table 1 of the HCCL RHD article: fold r = P - 2^floor(log P)
 *    part1 ranks, halving/doubling exchanges over the power-of-two core,
 *    copy back to the folded ranks.
 *  - Pipeline: "AllGather 算子的 Pipeline 时序编排", "Rank0 视角" and Table 1
 *    of the HCCL Pipeline article: inter-server ring overlapped with an
 *    intra-server full mesh, p_inter steps per phase.
 *  - Broadcast: Table 1 of the HCCL RHD article, Broadcast row (root parity
 *    picks the part1 members, distance halving, one last send).
 *  - Plain hierarchical AllReduce: intra-server ReduceScatter, inter-server
 *    RHD AllReduce, intra-server AllGather (Pipeline article, "与其它分级算法
 *    的关系"; RHD article, "耗时模型解读").  Its floating-point association
 *    order (the RHD tree over servers of intra-server chains rotated from the
 *    local index) is a reading; parity unpinned beyond the definition,
 *    exactly-once contributions and the step / traffic counts.
 *
 * Model of execution.  A schedule is a list of messages.  A message
 * (step, kind, src, dst, seg) sends the PRE-STEP value of segment seg held by
 * rank src to rank dst; all messages of a step are simultaneous.  A COPY
 * overwrites dst's value; a REDUCE folds the message into dst's value as
 *     v <- m (+) v        (received operand on the left, as in the ring
 *                          pseudo-code's reduce_op(recv, local))
 * in the order the messages are listed.  With loops, every message of loop i
 * covers only the i-th slice of its segment; loops run one after another.
 *
 * Arithmetic, per element and per step (the ring pseudo-code's element-wise
 * reduce_op; bf16 kept in bf16 between steps, so every step rounds):
 *   int32 : sum and prod wrap modulo 2^32; max/min by signed compare.
 *   fp32  : IEEE binary32, round to nearest even, no FMA, no flush to zero.
 *   bf16  : widen both operands to binary32, apply the op there, round the
 *           result back to bf16 (nearest even) after every step.
 *   max/min of fp32/bf16 follow the IEEE 754 totalOrder predicate on the
 *           bit patterns (-0 < +0, NaNs ordered by sign and payload), so they
 *           are commutative and associative bit for bit.
 *   sym   : symbolic mode; every value is an expression-tree node, used to
 *           read off the association order each schedule implies.
 *
 * Parity of the Pipeline ReduceScatter / AllReduce association order: the
 * pages narrate only the Pipeline AllGather and call the other two
 * "symmetric".  The order used here (a lone intra-server mesh reduce, then
 * the inter-server chain starting at server s+1) is pinned by the definition,
 * by every rank contributing exactly once and by Table 1's step structure,
 * but no printed value fixes the floating-point order itself: for fp32/bf16
 * sum and prod of the Pipeline ReduceScatter / AllReduce, parity unpinned
 * beyond those checks.
 *
 * Built with -O2 -ffp-contract=off and no fast-math (see build.py).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <stdio.h>

#define ORC_MAX_P 256

enum { ORC_RING = 0, ORC_RHD = 1, ORC_PIPE = 2, ORC_HIER = 3 };
enum { ORC_AR = 0, ORC_RS = 1, ORC_AG = 2, ORC_BCAST = 3 };
enum { ORC_I32 = 0, ORC_F32 = 1, ORC_BF16 = 2, ORC_SYM = 3 };
enum { ORC_SUM = 0, ORC_PROD = 1, ORC_MAX = 2, ORC_MIN = 3 };
enum { ORC_REDUCE = 0, ORC_COPY = 1 };

/* One message of the schedule, as exported to the test suite. */
typedef struct {
    int32_t loop;   /* loop index (slice of every segment) */
    int32_t step;   /* step index inside the loop */
    int32_t kind;   /* ORC_REDUCE or ORC_COPY */
    int32_t src;    /* sending rank */
    int32_t dst;    /* receiving rank */
    int32_t seg;    /* segment index */
    int64_t lo;     /* first element (absolute index in the rank vector) */
    int64_t hi;     /* one past the last element */
} orc_msg;

/* ------------------------------------------------------------------ */
/* small integer helpers                                               */
/* ------------------------------------------------------------------ */
static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
static int mod_int(int a, int m) { int r = a % m; return r < 0 ? r + m : r; }

static int elem_size(int dtype) {
    switch (dtype) {
    case ORC_I32: return 4;
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_SYM: return 4; /* symbolic values are laid out like a 4-byte type */
    default: return 0;
    }
}

/* largest power of two not above p (p >= 1) */
static int pow2_floor(int p) { int q = 1; while (q * 2 <= p) q *= 2; return q; }
static int log2_exact(int q) { int t = 0; while ((1 << t) < q) t++; return t; }

/* ------------------------------------------------------------------ */
/* segment layout                                                      */
/* ------------------------------------------------------------------ */
/*
 * Number of segments S: P for Ring, Pipeline and RHD ReduceScatter/AllGather
 * (one per rank: "数据向量被划分为P个等长块"); the power-of-two core size p' for
 * the RHD AllReduce, whose halving rounds split the vector among p' ranks.
 *
 * Segment length: the ring pseudo-code takes elem_count/rank_num, the Python
 * ring takes the ceiling, and the same section asks for chunk boundaries on
 * the DMA granule.  Reading used: L = ceil(n / S) rounded up to a multiple of
 * 16 bytes; segment k = [min(kL, n), min((k+1)L, n)).  Trailing segments may
 * be short or empty.
 */
int orc_num_segments(int algo, int coll, int P, int p_intra) {
    if (P < 1) return 0;
    if (coll == ORC_BCAST) return 1;  /* the whole vector moves as one block */
    if (algo == ORC_RHD && coll == ORC_AR) return pow2_floor(P);
    if (algo == ORC_HIER) {
        /* p_intra intra-server segments, each cut into the p' blocks of the
         * inter-server RHD over the P / p_intra servers */
        if (p_intra < 1 || P % p_intra) return 0;
        return p_intra * pow2_floor(P / p_intra);
    }
    return P;
}

int64_t orc_seg_stride(int algo, int coll, int P, int p_intra, int64_t n, int dtype) {
    int S = orc_num_segments(algo, coll, P, p_intra);
    int64_t A = 16 / elem_size(dtype);
    if (S <= 0 || n <= 0) return 0;
    return ceil_div64(ceil_div64(n, S), A) * A;
}

static void seg_range(int64_t L, int64_t n, int k, int64_t* lo, int64_t* hi) {
    *lo = min64((int64_t)k * L, n);
    *hi = min64((int64_t)(k + 1) * L, n);
}

int orc_segment(int algo, int coll, int P, int p_intra, int64_t n, int dtype, int k,
                int64_t* off, int64_t* len) {
    int S = orc_num_segments(algo, coll, P, p_intra);
    if (k < 0 || k >= S) return -1;
    int64_t L = orc_seg_stride(algo, coll, P, p_intra, n, dtype);
    int64_t lo, hi;
    seg_range(L, n, k, &lo, &hi);
    *off = lo;
    *len = hi - lo;
    return 0;
}

/* ------------------------------------------------------------------ */
/* loop / tail slicer                                                  */
/* ------------------------------------------------------------------ */
/*
 * The Pipeline article's OrchestrateLoop derives maxCountPerLoop from the
 * scratch limit maxTmpMemSize_, then loopTimes, and handles the tail slice on
 * its own.  The pages give no formula.  Reading used: with a byte limit Sb per
 * loop, every rank holds `slots` segment slices of c elements for each of the
 * P peers:   c = align_down(Sb / (P * slots * b), 128 / b),
 * slots = 1 (Ring), ceil(P/2) (RHD), p_intra - 1 (Pipeline and the plain
 * hierarchical AllReduce, at least 1).
 * The 128-byte alignment is the DMA granule of the AllReduce section.
 * Sb == 0 means a single loop.  Loop i covers [i*c, min((i+1)*c, len_k)) of
 * every segment k; the last loop is the tail.
 */
int orc_slicer(int algo, int coll, int P, int p_intra, int64_t n, int dtype,
               int64_t loop_bytes, int64_t* chunk, int* loops, int64_t* tail) {
    int64_t L = orc_seg_stride(algo, coll, P, p_intra, n, dtype);
    int b = elem_size(dtype);
    if (L <= 0 || loop_bytes <= 0) {
        *chunk = L; *loops = 1; *tail = L;
        return 0;
    }
    int64_t slots = 1;
    if (algo == ORC_RHD) slots = (P + 1) / 2;
    if (algo == ORC_PIPE || algo == ORC_HIER) slots = (p_intra - 1 > 1) ? (p_intra - 1) : 1;
    int64_t granule = 128 / b;
    int64_t c = loop_bytes / ((int64_t)P * slots * b);
    c = (c / granule) * granule;
    if (c < granule) c = granule;
    if (c >= L) {
        *chunk = L; *loops = 1; *tail = L;
        return 0;
    }
    int nl = (int)ceil_div64(L, c);
    *chunk = c;
    *loops = nl;
    *tail = L - (int64_t)(nl - 1) * c;
    return 0;
}

/* ------------------------------------------------------------------ */
/* schedule generators                                                 */
/* ------------------------------------------------------------------ */
typedef struct {
    int32_t step, kind, src, dst, seg;
} proto_msg;

typedef struct {
    proto_msg* v;
    int64_t n, cap;
    int nsteps;      /* steps used so far */
    int step_open;   /* messages were pushed into the current step */
} proto_vec;

static int pv_push(proto_vec* pv, int kind, int src, int dst, int seg) {
    if (pv->n == pv->cap) {
        int64_t nc = pv->cap ? pv->cap * 2 : 1024;
        proto_msg* nv = (proto_msg*)realloc(pv->v, (size_t)nc * sizeof(proto_msg));
        if (!nv) return -1;
        pv->v = nv;
        pv->cap = nc;
    }
    proto_msg m;
    m.step = pv->nsteps;
    m.kind = kind;
    m.src = src;
    m.dst = dst;
    m.seg = seg;
    pv->v[pv->n++] = m;
    pv->step_open = 1;
    return 0;
}

/* close the current step; a step without messages is not counted */
static void pv_end_step(proto_vec* pv) {
    if (pv->step_open) pv->nsteps++;
    pv->step_open = 0;
}

/*
 * Ring.  Reading of the two ring descriptions (the pseudo-code and the prose
 * of the AllReduce section disagree by one in the segment labels): at
 * reduce step s = 0..P-2 rank q sends segment (q-s-1) mod P to rank q+1, which
 * folds it into its own copy; so segment k's chain starts at rank k+1 and
 * ends at its owner k ("第i个设备拥有第i段").  At copy step s = 0..P-2 rank q
 * sends segment (q-s) mod P to rank q+1, starting with the segment it owns.
 */
static int gen_ring(proto_vec* pv, int coll, int P) {
    if (coll == ORC_AR || coll == ORC_RS) {
        for (int s = 0; s + 1 < P; s++) {
            for (int q = 0; q < P; q++)
                if (pv_push(pv, ORC_REDUCE, q, mod_int(q + 1, P), mod_int(q - s - 1, P))) return -1;
            pv_end_step(pv);
        }
    }
    if (coll == ORC_AR || coll == ORC_AG) {
        for (int s = 0; s + 1 < P; s++) {
            for (int q = 0; q < P; q++)
                if (pv_push(pv, ORC_COPY, q, mod_int(q + 1, P), mod_int(q - s, P))) return -1;
            pv_end_step(pv);
        }
    }
    return 0;
}

/*
 * Recursive Halving-Doubling.
 * Non-power-of-two P: r = P - p', p' = 2^floor(log2 P).  Part1 = ranks
 * 0..2r-1; odd rank 2i+1 folds into even rank 2i (the 5-rank example folds
 * rank1 into rank0).  Virtual rank of rank 2i (i < r) is i; of rank q >= 2r is
 * q - r.
 * AllReduce: partner = v XOR 2^t for t = 0,1,.. (lowest bit first); each
 * round halves the current window of p' blocks, the rank whose bit t is 0
 * keeping the lower half; doubling rounds run t back down and copy the owned
 * window to the partner; the folded odd ranks get the full result last.
 * ReduceScatter: same partners; before round t rank v holds the blocks of all
 * virtual ranks w agreeing with v on bits 0..t-1 and sends the partner those
 * with bit t equal to the partner's, which keeps blocks in scatter order
 * (rank r ends with block r); virtual rank i < r owns blocks 2i and 2i+1 and
 * the last step gives block 2i+1 to rank 2i+1.
 * AllGather: the mirror of ReduceScatter with copies.
 */
static int rhd_real(int v, int r) { return v < r ? 2 * v : v + r; }

static int rhd_blocks(int w, int r, int* blk) {
    if (w < r) { blk[0] = 2 * w; blk[1] = 2 * w + 1; return 2; }
    blk[0] = w + r;
    return 1;
}

static int gen_rhd(proto_vec* pv, int coll, int P) {
    int pp = pow2_floor(P);
    int r = P - pp;
    int lg = log2_exact(pp);
    if (coll == ORC_AR) {
        int S = pp;
        if (r > 0) {
            for (int i = 0; i < r; i++)
                for (int k = 0; k < S; k++)
                    if (pv_push(pv, ORC_REDUCE, 2 * i + 1, 2 * i, k)) return -1;
            pv_end_step(pv);
        }
        int* wlo = (int*)malloc(sizeof(int) * pp);
        int* whi = (int*)malloc(sizeof(int) * pp);
        int* nlo = (int*)malloc(sizeof(int) * pp);
        int* nhi = (int*)malloc(sizeof(int) * pp);
        if (!wlo || !whi || !nlo || !nhi) { free(wlo); free(whi); free(nlo); free(nhi); return -1; }
        for (int v = 0; v < pp; v++) { wlo[v] = 0; whi[v] = S; }
        for (int t = 0; t < lg; t++) {
            for (int v = 0; v < pp; v++) {
                int u = v ^ (1 << t);
                int mid = (wlo[v] + whi[v]) / 2;
                int klo, khi, slo, shi;
                if (((v >> t) & 1) == 0) { klo = wlo[v]; khi = mid; slo = mid; shi = whi[v]; }
                else { klo = mid; khi = whi[v]; slo = wlo[v]; shi = mid; }
                for (int k = slo; k < shi; k++)
                    if (pv_push(pv, ORC_REDUCE, rhd_real(v, r), rhd_real(u, r), k)) goto fail;
                nlo[v] = klo;
                nhi[v] = khi;
            }
            memcpy(wlo, nlo, sizeof(int) * pp);
            memcpy(whi, nhi, sizeof(int) * pp);
            pv_end_step(pv);
        }
        for (int t = lg - 1; t >= 0; t--) {
            for (int v = 0; v < pp; v++) {
                int u = v ^ (1 << t);
                for (int k = wlo[v]; k < whi[v]; k++)
                    if (pv_push(pv, ORC_COPY, rhd_real(v, r), rhd_real(u, r), k)) goto fail;
                nlo[v] = wlo[v] < wlo[u] ? wlo[v] : wlo[u];
                nhi[v] = whi[v] > whi[u] ? whi[v] : whi[u];
            }
            memcpy(wlo, nlo, sizeof(int) * pp);
            memcpy(whi, nhi, sizeof(int) * pp);
            pv_end_step(pv);
        }
        free(wlo); free(whi); free(nlo); free(nhi);
        if (r > 0) {
            for (int i = 0; i < r; i++)
                for (int k = 0; k < S; k++)
                    if (pv_push(pv, ORC_COPY, 2 * i, 2 * i + 1, k)) return -1;
            pv_end_step(pv);
        }
        return 0;
    fail:
        free(wlo); free(whi); free(nlo); free(nhi);
        return -1;
    }
    if (coll == ORC_RS) {
        if (r > 0) {
            for (int i = 0; i < r; i++)
                for (int k = 0; k < P; k++)
                    if (pv_push(pv, ORC_REDUCE, 2 * i + 1, 2 * i, k)) return -1;
            pv_end_step(pv);
        }
        for (int t = 0; t < lg; t++) {
            int low = (1 << t) - 1;
            for (int v = 0; v < pp; v++) {
                int u = v ^ (1 << t);
                for (int w = 0; w < pp; w++) {
                    if ((w & low) != (v & low)) continue;
                    if (((w >> t) & 1) != ((u >> t) & 1)) continue;
                    int blk[2];
                    int nb = rhd_blocks(w, r, blk);
                    for (int j = 0; j < nb; j++)
                        if (pv_push(pv, ORC_REDUCE, rhd_real(v, r), rhd_real(u, r), blk[j])) return -1;
                }
            }
            pv_end_step(pv);
        }
        if (r > 0) {
            for (int i = 0; i < r; i++)
                if (pv_push(pv, ORC_COPY, 2 * i, 2 * i + 1, 2 * i + 1)) return -1;
            pv_end_step(pv);
        }
        return 0;
    }
    /* AllGather */
    if (r > 0) {
        for (int i = 0; i < r; i++)
            if (pv_push(pv, ORC_COPY, 2 * i + 1, 2 * i, 2 * i + 1)) return -1;
        pv_end_step(pv);
    }
    for (int t = lg - 1; t >= 0; t--) {
        int low = (1 << (t + 1)) - 1;
        for (int v = 0; v < pp; v++) {
            int u = v ^ (1 << t);
            for (int w = 0; w < pp; w++) {
                if ((w & low) != (v & low)) continue;
                int blk[2];
                int nb = rhd_blocks(w, r, blk);
                for (int j = 0; j < nb; j++)
                    if (pv_push(pv, ORC_COPY, rhd_real(v, r), rhd_real(u, r), blk[j])) return -1;
            }
        }
        pv_end_step(pv);
    }
    if (r > 0) {
        for (int i = 0; i < r; i++)
            for (int k = 0; k < P; k++)
                if (pv_push(pv, ORC_COPY, 2 * i, 2 * i + 1, k)) return -1;
        pv_end_step(pv);
    }
    return 0;
}

/*
 * RHD Broadcast (Table 1 of the RHD article, Broadcast row): the root's
 * parity decides whether the even or the odd rank of each part1 pair
 * (2i, 2i+1), i < r, joins the power-of-two block; inside the block the data
 * spreads by distance halving (partner = v XOR p'/2, then p'/4, ..., 1, every
 * holder sending to its partner); one last step sends from each part1 block
 * member to its pair partner.  ceil(log2 P) steps, each moving n elements.
 */
static int gen_rhd_bcast(proto_vec* pv, int P, int root) {
    int pp = pow2_floor(P);
    int r = P - pp;
    int par = root & 1;
    int vroot = root < 2 * r ? root / 2 : root - r;
    char* have = (char*)calloc((size_t)pp, 1);
    char* next = (char*)calloc((size_t)pp, 1);
    if (!have || !next) { free(have); free(next); return -1; }
    have[vroot] = 1;
    for (int d = pp / 2; d >= 1; d /= 2) {
        memcpy(next, have, (size_t)pp);
        for (int v = 0; v < pp; v++) {
            if (!have[v]) continue;
            int u = v ^ d;
            int rv = v < r ? 2 * v + par : v + r;
            int ru = u < r ? 2 * u + par : u + r;
            if (pv_push(pv, ORC_COPY, rv, ru, 0)) { free(have); free(next); return -1; }
            next[u] = 1;
        }
        memcpy(have, next, (size_t)pp);
        pv_end_step(pv);
    }
    free(have);
    free(next);
    if (r > 0) {
        for (int i = 0; i < r; i++)
            if (pv_push(pv, ORC_COPY, 2 * i + par, 2 * i + 1 - par, 0)) return -1;
        pv_end_step(pv);
    }
    return 0;
}

/*
 * Hierarchical Pipeline, P = p_inter x p_intra, rank = s * p_intra + l
 * (server-major), inter ring s -> s+1 among ranks of equal local index l.
 * AllGather (the narrated case): at step t = 1..p_inter every rank (s,l)
 * forwards the block it holds since step t-1 (its own block at t = 1) along
 * the ring to (s+1,l) (steps 1..p_inter-1 only) and to every other rank of its
 * server; the last step is the lone intra-server transfer.
 * ReduceScatter (the pages only say it is symmetric; reading used): the chain
 * of block (b,l) starts at server b+1 and ends at owner b.  Step 1 is a lone
 * intra-server mesh reduce; at step t the rank (b+t, l) mesh-reduces block
 * (b,l) from the other ranks of its server, in local order l+1, l+2, .., and
 * then folds in the partial arriving on the ring from (b+t-1, l).
 */
static int gen_pipe(proto_vec* pv, int coll, int P, int p_intra) {
    int pin = p_intra;
    int pout = P / pin;
    if (coll == ORC_AR || coll == ORC_RS) {
        for (int t = 1; t <= pout; t++) {
            for (int s = 0; s < pout; s++) {
                for (int l = 0; l < pin; l++) {
                    int b = mod_int(s - t, pout);
                    int seg = b * pin + l;
                    int dst = s * pin + l;
                    for (int j = 1; j < pin; j++)
                        if (pv_push(pv, ORC_REDUCE, s * pin + mod_int(l + j, pin), dst, seg)) return -1;
                    if (t >= 2)
                        if (pv_push(pv, ORC_REDUCE, mod_int(s - 1, pout) * pin + l, dst, seg)) return -1;
                }
            }
            pv_end_step(pv);
        }
    }
    if (coll == ORC_AR || coll == ORC_AG) {
        for (int t = 1; t <= pout; t++) {
            for (int s = 0; s < pout; s++) {
                for (int l = 0; l < pin; l++) {
                    int src = s * pin + l;
                    int seg = mod_int(s - t + 1, pout) * pin + l;
                    if (t <= pout - 1)
                        if (pv_push(pv, ORC_COPY, src, mod_int(s + 1, pout) * pin + l, seg)) return -1;
                    for (int j = 1; j < pin; j++)
                        if (pv_push(pv, ORC_COPY, src, s * pin + mod_int(l + j, pin), seg)) return -1;
                }
            }
            pv_end_step(pv);
        }
    }
    return 0;
}

/*
 * Plain hierarchical AllReduce (the Pipeline article's "与其它分级算法的关系":
 * Server 内 ReduceScatter -> Server 间 AllReduce -> Server 内 AllGather; the
 * RHD article's "耗时模型解读" puts RHD at the inter-server level and
 * Mesh / Ring inside the server).  Reading used: P = p_inter x p_intra,
 * rank = s * p_intra + l; the intra-server phases are full-mesh steps; the
 * inter-server AllReduce is the RHD AllReduce (fold, halving, doubling,
 * unfold) among the ranks of equal local index l, on intra segment l.
 * Segments: intra segment l is made of the p' blocks l*p' .. l*p' + p' - 1
 * (p' = 2^floor(log2 p_inter)).
 *  step A (if p_intra > 1): (s,l) receives every block of intra segment l
 *    from (s,l+1), (s,l+2), ... and folds them into its own;
 *  steps B: RHD AllReduce over servers within each local index;
 *  step C (if p_intra > 1): (s,l) copies intra segment l to every (s,l').
 */
static int gen_hier(proto_vec* pv, int P, int pin) {
    const int pout = P / pin;
    const int pp = pow2_floor(pout);
    const int r = pout - pp;
    const int lg = log2_exact(pp);
    #define HR(s, l) ((s) * pin + (l))
    #define SV(v) ((v) < r ? 2 * (v) : (v) + r)
    if (pin > 1) {
        for (int s = 0; s < pout; s++)
            for (int l = 0; l < pin; l++)
                for (int j = 1; j < pin; j++)
                    for (int b = 0; b < pp; b++)
                        if (pv_push(pv, ORC_REDUCE, HR(s, mod_int(l + j, pin)), HR(s, l), l * pp + b))
                            return -1;
        pv_end_step(pv);
    }
    if (r > 0) {
        for (int l = 0; l < pin; l++)
            for (int i = 0; i < r; i++)
                for (int b = 0; b < pp; b++)
                    if (pv_push(pv, ORC_REDUCE, HR(2 * i + 1, l), HR(2 * i, l), l * pp + b)) return -1;
        pv_end_step(pv);
    }
    int* wlo = (int*)malloc(sizeof(int) * pp);
    int* whi = (int*)malloc(sizeof(int) * pp);
    int* nlo = (int*)malloc(sizeof(int) * pp);
    int* nhi = (int*)malloc(sizeof(int) * pp);
    if (!wlo || !whi || !nlo || !nhi) { free(wlo); free(whi); free(nlo); free(nhi); return -1; }
    int rc = 0;
    for (int v = 0; v < pp; v++) { wlo[v] = 0; whi[v] = pp; }
    for (int t = 0; t < lg && !rc; t++) {
        for (int v = 0; v < pp; v++) {
            int u = v ^ (1 << t), mid = (wlo[v] + whi[v]) / 2;
            int keep_low = ((v >> t) & 1) == 0;
            int glo = keep_low ? mid : wlo[v], ghi = keep_low ? whi[v] : mid;
            for (int l = 0; l < pin && !rc; l++)
                for (int k = glo; k < ghi && !rc; k++)
                    rc = pv_push(pv, ORC_REDUCE, HR(SV(v), l), HR(SV(u), l), l * pp + k);
            nlo[v] = keep_low ? wlo[v] : mid;
            nhi[v] = keep_low ? mid : whi[v];
        }
        memcpy(wlo, nlo, sizeof(int) * pp);
        memcpy(whi, nhi, sizeof(int) * pp);
        pv_end_step(pv);
    }
    for (int t = lg - 1; t >= 0 && !rc; t--) {
        for (int v = 0; v < pp; v++) {
            int u = v ^ (1 << t);
            for (int l = 0; l < pin && !rc; l++)
                for (int k = wlo[v]; k < whi[v] && !rc; k++)
                    rc = pv_push(pv, ORC_COPY, HR(SV(v), l), HR(SV(u), l), l * pp + k);
            nlo[v] = wlo[v] < wlo[u] ? wlo[v] : wlo[u];
            nhi[v] = whi[v] > whi[u] ? whi[v] : whi[u];
        }
        memcpy(wlo, nlo, sizeof(int) * pp);
        memcpy(whi, nhi, sizeof(int) * pp);
        pv_end_step(pv);
    }
    free(wlo); free(whi); free(nlo); free(nhi);
    if (rc) return -1;
    if (r > 0) {
        for (int l = 0; l < pin; l++)
            for (int i = 0; i < r; i++)
                for (int b = 0; b < pp; b++)
                    if (pv_push(pv, ORC_COPY, HR(2 * i, l), HR(2 * i + 1, l), l * pp + b)) return -1;
        pv_end_step(pv);
    }
    if (pin > 1) {
        for (int s = 0; s < pout; s++)
            for (int l = 0; l < pin; l++)
                for (int j = 1; j < pin; j++)
                    for (int b = 0; b < pp; b++)
                        if (pv_push(pv, ORC_COPY, HR(s, l), HR(s, mod_int(l + j, pin)), l * pp + b))
                            return -1;
        pv_end_step(pv);
    }
    #undef HR
    #undef SV
    return 0;
}

static int check_args(int algo, int coll, int P, int p_intra, int64_t n, int dtype) {
    if (algo < ORC_RING || algo > ORC_HIER) return -1;
    if (algo == ORC_HIER && (coll != ORC_AR || p_intra < 1 || P % p_intra)) return -1;
    if (coll < ORC_AR || coll > ORC_BCAST) return -1;
    if (coll == ORC_BCAST && algo != ORC_RHD) return -1;  /* only the RHD broadcast is described */
    if (P < 1 || P > ORC_MAX_P) return -1;
    if (n < 0) return -1;
    if (elem_size(dtype) == 0) return -1;
    if (algo == ORC_PIPE && (p_intra < 1 || P % p_intra != 0)) return -1;
    return 0;
}

/*
 * Build the full message list: the loop-independent step list repeated per
 * loop, every message restricted to the loop's slice of its segment (messages
 * whose slice is empty are dropped).  Returns the number of messages, or -1.
 * The caller frees *out with orc_free.
 */
static int64_t build_schedule(int algo, int coll, int P, int p_intra, int root, int64_t n,
                              int dtype, int64_t loop_bytes, orc_msg** out, int* steps_per_loop,
                              int* nloops) {
    *out = NULL;
    if (check_args(algo, coll, P, p_intra, n, dtype)) return -1;
    if (root < 0 || root >= P) return -1;
    proto_vec pv = {0};
    int rc;
    if (coll == ORC_BCAST) rc = gen_rhd_bcast(&pv, P, root);
    else if (algo == ORC_HIER) rc = gen_hier(&pv, P, p_intra);
    else if (algo == ORC_RING) rc = gen_ring(&pv, coll, P);
    else if (algo == ORC_RHD) rc = gen_rhd(&pv, coll, P);
    else rc = gen_pipe(&pv, coll, P, p_intra);
    if (rc) { free(pv.v); return -1; }
    int64_t c, tail;
    int loops;
    orc_slicer(algo, coll, P, p_intra, n, dtype, loop_bytes, &c, &loops, &tail);
    int64_t L = orc_seg_stride(algo, coll, P, p_intra, n, dtype);
    int64_t cap = pv.n * (int64_t)loops;
    orc_msg* v = (orc_msg*)malloc(sizeof(orc_msg) * (size_t)(cap > 0 ? cap : 1));
    if (!v) { free(pv.v); return -1; }
    int64_t m = 0;
    for (int i = 0; i < loops; i++) {
        for (int64_t q = 0; q < pv.n; q++) {
            proto_msg* pm = &pv.v[q];
            int64_t slo, shi;
            seg_range(L, n, pm->seg, &slo, &shi);
            int64_t a = slo + (int64_t)i * c;
            int64_t b = min64(slo + (int64_t)(i + 1) * c, shi);
            if (a >= b) continue;
            orc_msg mm;
            mm.loop = i;
            mm.step = pm->step;
            mm.kind = pm->kind;
            mm.src = pm->src;
            mm.dst = pm->dst;
            mm.seg = pm->seg;
            mm.lo = a;
            mm.hi = b;
            v[m++] = mm;
        }
    }
    *steps_per_loop = pv.nsteps;
    *nloops = loops;
    free(pv.v);
    *out = v;
    return m;
}

/* Exported: the schedule as a message list (test suite reads it).  root is
 * used by the Broadcast only. */
int64_t orc_schedule(int algo, int coll, int P, int p_intra, int root, int64_t n, int dtype,
                     int64_t loop_bytes, orc_msg** out, int* steps_per_loop, int* nloops) {
    return build_schedule(algo, coll, P, p_intra, root, n, dtype, loop_bytes, out, steps_per_loop,
                          nloops);
}

void orc_free(void* p) { free(p); }

/* ------------------------------------------------------------------ */
/* arithmetic                                                          */
/* ------------------------------------------------------------------ */
static float f32_of_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_of_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the top half of a binary32 */
static float bf16_to_f32(uint16_t h) { return f32_of_bits((uint32_t)h << 16); }

/* binary32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u = bits_of_f32(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* IEEE 754 totalOrder key: unsigned comparison of keys = totalOrder */
static uint32_t order_key32(uint32_t u) { return (u & 0x80000000u) ? ~u : (u | 0x80000000u); }
static uint16_t order_key16(uint16_t u) {
    return (uint16_t)((u & 0x8000u) ? (uint16_t)~u : (uint16_t)(u | 0x8000u));
}

/* symbolic expression pool: ids < ORC_MAX_P are leaves X_id, ORC_MAX_P is
 * the "never written" marker, larger ids are (+) nodes */
#define SYM_POISON ORC_MAX_P
#define SYM_BASE (ORC_MAX_P + 1)
typedef struct { int64_t a, b; } sym_node;
static sym_node* g_sym = NULL;
static int64_t g_sym_n = 0, g_sym_cap = 0;

static int64_t sym_make(int64_t a, int64_t b) {
    if (g_sym_n == g_sym_cap) {
        int64_t nc = g_sym_cap ? g_sym_cap * 2 : 4096;
        sym_node* nv = (sym_node*)realloc(g_sym, (size_t)nc * sizeof(sym_node));
        if (!nv) return -1;
        g_sym = nv;
        g_sym_cap = nc;
    }
    g_sym[g_sym_n].a = a;
    g_sym[g_sym_n].b = b;
    return SYM_BASE + g_sym_n++;
}

void orc_sym_reset(void) { g_sym_n = 0; }

static uint64_t combine(int dtype, int op, uint64_t a, uint64_t b) {
    switch (dtype) {
    case ORC_I32: {
        uint32_t x = (uint32_t)a, y = (uint32_t)b;
        int32_t sx = (int32_t)x, sy = (int32_t)y;
        switch (op) {
        case ORC_SUM: return (uint32_t)(x + y);
        case ORC_PROD: return (uint32_t)(x * y);
        case ORC_MAX: return sx < sy ? y : x;
        default: return sy < sx ? y : x;
        }
    }
    case ORC_F32: {
        uint32_t x = (uint32_t)a, y = (uint32_t)b;
        switch (op) {
        case ORC_SUM: return bits_of_f32(f32_of_bits(x) + f32_of_bits(y));
        case ORC_PROD: return bits_of_f32(f32_of_bits(x) * f32_of_bits(y));
        case ORC_MAX: return order_key32(x) < order_key32(y) ? y : x;
        default: return order_key32(y) < order_key32(x) ? y : x;
        }
    }
    case ORC_BF16: {
        uint16_t x = (uint16_t)a, y = (uint16_t)b;
        switch (op) {
        case ORC_SUM: return orc_f32_to_bf16(bf16_to_f32(x) + bf16_to_f32(y));
        case ORC_PROD: return orc_f32_to_bf16(bf16_to_f32(x) * bf16_to_f32(y));
        case ORC_MAX: return order_key16(x) < order_key16(y) ? y : x;
        default: return order_key16(y) < order_key16(x) ? y : x;
        }
    }
    default:
        return (uint64_t)sym_make((int64_t)a, (int64_t)b);
    }
}

static uint64_t load_raw(int dtype, const void* X, int64_t idx) {
    if (dtype == ORC_BF16) return ((const uint16_t*)X)[idx];
    return ((const uint32_t*)X)[idx];
}

static void store_raw(int dtype, void* Y, int64_t idx, uint64_t v) {
    if (dtype == ORC_BF16) ((uint16_t*)Y)[idx] = (uint16_t)v;
    else if (dtype == ORC_SYM) ((int64_t*)Y)[idx] = (int64_t)v;
    else ((uint32_t*)Y)[idx] = (uint32_t)v;
}

/* first index i in sorted J with J[i] >= x */
static int64_t lower_bound(const int64_t* J, int64_t nJ, int64_t x) {
    int64_t lo = 0, hi = nJ;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (J[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

/*
 * Step-by-step replay.
 *   X : P rank vectors of n elements, row-major (ignored for ORC_SYM)
 *   J : sorted element indices to follow (NULL = all 0..n-1), nJ of them
 *   Y : P x nJ values after the schedule (int64 node ids for ORC_SYM)
 * AllGather: rank r starts with segment r of X[r]; its other elements start
 * as X[r] too (ORC_SYM: as the "never written" marker), so an element the
 * schedule fails to deliver is visible.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
static int replay_impl(int algo, int coll, int P, int p_intra, int root, int64_t n, int dtype,
                       int ldtype, int op, int64_t loop_bytes, const void* X, const int64_t* J,
                       int64_t nJ, void* Y) {
    if (check_args(algo, coll, P, p_intra, n, ldtype)) return -1;
    if (ldtype == ORC_SYM) return -1;
    if (op < ORC_SUM || op > ORC_MIN) return -1;
    int64_t* Jall = NULL;
    if (!J) {
        nJ = n;
        Jall = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
        if (!Jall) return -1;
        for (int64_t i = 0; i < n; i++) Jall[i] = i;
        J = Jall;
    }
    for (int64_t i = 0; i + 1 < nJ; i++)
        if (J[i] >= J[i + 1]) { free(Jall); return -1; }
    for (int64_t i = 0; i < nJ; i++)
        if (J[i] < 0 || J[i] >= n) { free(Jall); return -1; }

    orc_msg* msgs = NULL;
    int spl = 0, loops = 0;
    int64_t nm = build_schedule(algo, coll, P, p_intra, root, n, ldtype, loop_bytes, &msgs, &spl,
                                &loops);
    if (nm < 0) { free(Jall); return -1; }

    size_t cells = (size_t)P * (size_t)(nJ > 0 ? nJ : 1);
    uint64_t* cur = (uint64_t*)malloc(sizeof(uint64_t) * cells);
    uint64_t* nxt = (uint64_t*)malloc(sizeof(uint64_t) * cells);
    if (!cur || !nxt) { free(cur); free(nxt); free(msgs); free(Jall); return -1; }

    int64_t L = orc_seg_stride(algo, coll, P, p_intra, n, ldtype);
    for (int q = 0; q < P; q++) {
        for (int64_t i = 0; i < nJ; i++) {
            uint64_t v;
            if (dtype == ORC_SYM) {
                v = (uint64_t)q;
                if (coll == ORC_AG) {
                    int64_t slo, shi;
                    seg_range(L, n, q, &slo, &shi);
                    if (J[i] < slo || J[i] >= shi) v = SYM_POISON;
                }
                if (coll == ORC_BCAST && q != root) v = SYM_POISON;
            } else {
                v = load_raw(dtype, X, (int64_t)q * n + J[i]);
            }
            cur[(size_t)q * nJ + i] = v;
        }
    }

    /* messages are grouped by (loop, step) in generation order */
    int64_t a = 0;
    while (a < nm) {
        int64_t b = a;
        while (b < nm && msgs[b].loop == msgs[a].loop && msgs[b].step == msgs[a].step) b++;
        memcpy(nxt, cur, sizeof(uint64_t) * cells);
        for (int64_t q = a; q < b; q++) {
            orc_msg* m = &msgs[q];
            int64_t i = lower_bound(J, nJ, m->lo);
            for (; i < nJ && J[i] < m->hi; i++) {
                uint64_t mv = cur[(size_t)m->src * nJ + i];
                uint64_t* dv = &nxt[(size_t)m->dst * nJ + i];
                if (m->kind == ORC_COPY) *dv = mv;
                else *dv = combine(dtype, op, mv, *dv);
            }
        }
        uint64_t* t = cur; cur = nxt; nxt = t;
        a = b;
    }

    for (int q = 0; q < P; q++)
        for (int64_t i = 0; i < nJ; i++)
            store_raw(dtype, Y, (int64_t)q * nJ + i, cur[(size_t)q * nJ + i]);

    free(cur); free(nxt); free(msgs); free(Jall);
    return 0;
}

int orc_replay(int algo, int coll, int P, int p_intra, int root, int64_t n, int dtype, int op,
               int64_t loop_bytes, const void* X, const int64_t* J, int64_t nJ, void* Y) {
    if (dtype == ORC_SYM) return -1;
    return replay_impl(algo, coll, P, p_intra, root, n, dtype, dtype, op, loop_bytes, X, J, nJ, Y);
}

/* Symbolic replay: the schedule of a layout dtype (its 16-byte segment
 * rounding), every value an expression node; Y holds P x nJ int64 node ids
 * (read them back with orc_sym_string / orc_sym_leaves). */
int orc_replay_sym(int algo, int coll, int P, int p_intra, int root, int64_t n, int layout_dtype,
                   int64_t loop_bytes, const int64_t* J, int64_t nJ, int64_t* Y) {
    return replay_impl(algo, coll, P, p_intra, root, n, ORC_SYM, layout_dtype, ORC_SUM, loop_bytes,
                       NULL, J, nJ, Y);
}

/* ------------------------------------------------------------------ */
/* symbolic read-back                                                  */
/* ------------------------------------------------------------------ */
static int64_t put_char(char* buf, int64_t cap, int64_t pos, char c) {
    if (pos < cap - 1) buf[pos] = c;
    return pos + 1;
}

static int64_t sym_str_rec(int64_t id, char* buf, int64_t cap, int64_t pos) {
    if (id < SYM_BASE) {
        char tmp[32];
        int k = (id == SYM_POISON) ? snprintf(tmp, sizeof tmp, "?") : snprintf(tmp, sizeof tmp, "X%d", (int)id);
        for (int j = 0; j < k; j++) pos = put_char(buf, cap, pos, tmp[j]);
        return pos;
    }
    sym_node nd = g_sym[id - SYM_BASE];
    pos = put_char(buf, cap, pos, '(');
    pos = sym_str_rec(nd.a, buf, cap, pos);
    pos = put_char(buf, cap, pos, '+');
    pos = sym_str_rec(nd.b, buf, cap, pos);
    return put_char(buf, cap, pos, ')');
}

/* Writes the expression of node id ("(A+B)", leaves "X3", "?" = never
 * written) into buf, NUL-terminated; returns the full length needed. */
int64_t orc_sym_string(int64_t id, char* buf, int64_t cap) {
    int64_t len = sym_str_rec(id, buf, cap, 0);
    if (cap > 0) buf[len < cap ? len : cap - 1] = '\0';
    return len;
}

/* Counts how often each leaf occurs in node id: counts[0..ORC_MAX_P]
 * (index ORC_MAX_P counts "never written" markers).  Iterative walk. */
int orc_sym_leaves(int64_t id, int64_t* counts) {
    int64_t cap = 1024, top = 0;
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
    if (!st) return -1;
    st[top++] = id;
    while (top > 0) {
        int64_t x = st[--top];
        if (x < SYM_BASE) { counts[x]++; continue; }
        if (top + 2 > cap) {
            cap *= 2;
            int64_t* ns = (int64_t*)realloc(st, sizeof(int64_t) * (size_t)cap);
            if (!ns) { free(st); return -1; }
            st = ns;
        }
        st[top++] = g_sym[x - SYM_BASE].a;
        st[top++] = g_sym[x - SYM_BASE].b;
    }
    free(st);
    return 0;
}

/* ------------------------------------------------------------------ */
/* direct definition                                                   */
/* ------------------------------------------------------------------ */
/*
 * Y[j] = (+)_i X_i[j] straight from the definition.
 *  int32      : exact, wrapped to 32 bits (Y raw).
 *  max / min  : totalOrder over the raw bits (Y raw), any dtype.
 *  fp sum/prod: in binary64 over i = 0..P-1 (Y64); Y raw is not written.
 * Also returns, for fp sum, S1[j] = sum_i |X_i[j]| in binary64 (may be NULL),
 * the scale of the per-element error bound.
 */
int orc_direct(int dtype, int op, int P, int64_t n, const void* X, void* Y, double* Y64, double* S1) {
    if (P < 1 || n < 0 || dtype < ORC_I32 || dtype > ORC_BF16) return -1;
    for (int64_t j = 0; j < n; j++) {
        if (dtype == ORC_I32) {
            if (op == ORC_SUM || op == ORC_PROD) {
                uint32_t acc = (op == ORC_SUM) ? 0u : 1u;
                for (int i = 0; i < P; i++) {
                    uint32_t x = (uint32_t)load_raw(dtype, X, (int64_t)i * n + j);
                    acc = (op == ORC_SUM) ? acc + x : acc * x;
                }
                store_raw(dtype, Y, j, acc);
                if (Y64) {
                    double d = (op == ORC_SUM) ? 0.0 : 1.0;
                    for (int i = 0; i < P; i++) {
                        int32_t x = (int32_t)(uint32_t)load_raw(dtype, X, (int64_t)i * n + j);
                        d = (op == ORC_SUM) ? d + (double)x : d * (double)x;
                    }
                    Y64[j] = d;
                }
                continue;
            }
        }
        if (op == ORC_MAX || op == ORC_MIN) {
            uint64_t acc = load_raw(dtype, X, j);
            for (int i = 1; i < P; i++) {
                uint64_t x = load_raw(dtype, X, (int64_t)i * n + j);
                int take;
                if (dtype == ORC_I32) {
                    int32_t sa = (int32_t)(uint32_t)acc, sx = (int32_t)(uint32_t)x;
                    take = (op == ORC_MAX) ? (sx > sa) : (sx < sa);
                } else if (dtype == ORC_F32) {
                    uint32_t ka = order_key32((uint32_t)acc), kx = order_key32((uint32_t)x);
                    take = (op == ORC_MAX) ? (kx > ka) : (kx < ka);
                } else {
                    uint16_t ka = order_key16((uint16_t)acc), kx = order_key16((uint16_t)x);
                    take = (op == ORC_MAX) ? (kx > ka) : (kx < ka);
                }
                if (take) acc = x;
            }
            store_raw(dtype, Y, j, acc);
            continue;
        }
        double d = (op == ORC_SUM) ? 0.0 : 1.0, s1 = 0.0;
        for (int i = 0; i < P; i++) {
            uint64_t x = load_raw(dtype, X, (int64_t)i * n + j);
            double xv = (dtype == ORC_F32) ? (double)f32_of_bits((uint32_t)x) : (double)bf16_to_f32((uint16_t)x);
            if (op == ORC_SUM) d += xv; else d *= xv;
            s1 += xv < 0 ? -xv : xv;
        }
        if (Y64) Y64[j] = d;
        if (S1) S1[j] = s1;
    }
    return 0;
}
