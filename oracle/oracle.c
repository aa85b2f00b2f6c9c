/*
 * oracle.c -- plain, slow CPU oracle for collectives among N virtual ranks.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
 * baseline call this file.  It shares no code, header, table or constant with the
 * CUDA path; both sides receive the same seeded input bytes and nothing else.
 *
 * What it computes (one plain loop per definition, no blocking, no staging):
 *
 *  - All-reduce, reduce-scatter: every rank's buffer reduced element by element
 *    ("AI Systems Performance Engineering (3)", collective table: all-reduce row,
 *    reduce-scatter row).  The reduction ORDER is the ring's order.  A ring
 *    reduce-scatter hands the partial of chunk c from rank to rank; in the chunk
 *    arithmetic of RingARAlgorithm::getNextSendAddr (NCCL book, section 2.3
 *    "algorithm", Ring), rank r at stage s works on chunk (r + N - 1 - s) mod N, so
 *    chunk b starts at rank b+1 and is finished at rank b.  The element partial is
 *    therefore  acc = x[b+1]; acc = OP(acc, x[b+2]); ...; acc = OP(acc, x[b])  with
 *    every intermediate result rounded to the storage type (each hop stores the
 *    partial in the receiver's buffer in that type).
 *  - Block size for all-reduce: B = alignUp(ceil(count / N), 16 / elemSize)
 *    elements, the tail-chunk rule of the same getNextSendAddr; element e belongs to
 *    block floor(e / B).  For reduce-scatter block r is exactly the recvcount
 *    elements that rank r receives.
 *  - All-gather: recv_r = concat over s of send_s (collective table, all-gather row;
 *    the bootstrap ring AllGather of "NCCL Expert Course 17: Bootstrap and
 *    Communicator Init State Machine" moves the same slices).
 *  - Broadcast: recv_r = send_root (collective table, broadcast row).
 *  - All-to-all: rank i's j-th block goes to rank j's i-th block, a block transpose
 *    (collective table, all-to-all row); the variable-size form takes element
 *    counts and displacements per (sender, receiver).
 *  - Non-reducing collectives are byte copies whatever the data type (NCCL book,
 *    chapter 6, taskAppend: AllGather/Broadcast run as ncclInt8).
 *  - Reduce (to root): recv_root = the reduction of all ranks, every element in the
 *    ring order root+1, ..., root -- the order of a ring chain that ends at the root
 *    (collective table, reduce row; NCCL runs Reduce as such a chain).  Gather:
 *    recv_root = concat over s of send_s.  Scatter: recv_r = block r of send_root
 *    (collective table, gather and scatter rows).
 *  - Double binary tree all-reduce (NCCL book chapter 4, trees.cc ncclGetBtree /
 *    ncclGetDtree): the first half of the buffer is reduced up tree 0 (the binary tree
 *    rooted at rank 0 that ncclGetBtree builds from the ranks' lowest set bits), the
 *    second half up tree 1 (tree 0 mirrored, rank r -> N-1-r, for even N; shifted,
 *    r -> r+1, for odd N); every rank receives the root's result.  A node's partial is its
 *    own element, then OP with the partial of child d0, then with that of child d1.
 *  - Special cases: count 0 does nothing; N = 1 is a plain copy (taskAppend:
 *    count==0 returns at once, nRanks==1 runs a local one-rank reduction).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - prod/min/max and int32 are not on the pages (only SUM is).  Int32 sum and prod
 *    wrap modulo 2^32.  min keeps the running partial a unless (b < a); max keeps a
 *    unless (b > a); the comparison is made on exactly converted fp32 values and the
 *    selected element keeps its original bits.
 *  - fp16/bf16 sum and prod: both operands converted exactly to fp32, one fp32 op
 *    with round-to-nearest-even, then rounded to the storage type (RNE).
 *  - reduce-scatter with a fused epilogue: out = (float)acc * scale in fp32 (RNE),
 *    optionally rounded back to the input type.
 *
 * fp16/bf16 conversions are written here from the IEEE 754 binary16 and bfloat16
 * definitions; the unit tests pin them against torch's and numpy's converters.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no -ffast-math, no FMA contraction,
 * no flush-to-zero).  Every entry point returns 0 on success and a negative value for
 * bad arguments.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_I32 = 3 };
enum { ORC_SUM = 0, ORC_PROD = 1, ORC_MIN = 2, ORC_MAX = 3 };

/* ----------------------------------------------------------------------------- */
/* Scalar conversions from the format definitions.                                 */
/* ----------------------------------------------------------------------------- */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bfloat16 is the top half of a binary32. */
float orc_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* binary32 -> bfloat16, round to nearest, ties to even.  Dropping the low 16 bits
 * rounds up when they exceed half an ulp of the kept part, or equal it and the kept
 * part is odd; adding 0x7FFF plus the kept lsb and truncating does exactly that and
 * carries into the exponent (up to infinity) when the mantissa overflows. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u = f32_to_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);           /* NaN stays a quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
float orc_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t m = h & 0x3FFu;
    if (e == 0) {
        float v = ldexpf((float)m, -24);                 /* zero or subnormal: m * 2^-24, exact */
        return sign ? -v : v;
    }
    if (e == 31) return bits_to_f32(sign | 0x7F800000u | (m << 13));  /* inf / NaN */
    return bits_to_f32(sign | ((e - 15 + 127) << 23) | (m << 13));
}

/* Shift a significand right by sh bits, rounding to nearest, ties to even. */
static uint64_t shift_rne(uint64_t sig, int sh) {
    if (sh <= 0) return sig;
    if (sh >= 64) return 0;
    uint64_t kept = sig >> sh;
    uint64_t rem = sig & ((1ull << sh) - 1);
    uint64_t half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (kept & 1))) kept++;
    return kept;
}

uint16_t orc_f32_to_f16(float f) {
    uint32_t u = f32_to_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t fe = (u >> 23) & 0xFFu;
    uint32_t fm = u & 0x7FFFFFu;
    if (fe == 0xFF) return fm ? (uint16_t)(sign | 0x7E00u | (fm >> 13)) : (uint16_t)(sign | 0x7C00u);
    if (fe == 0) return sign;                             /* binary32 subnormals are < 2^-126 */
    int e = (int)fe - 127;                                /* value = 1.fm * 2^e */
    uint64_t sig = (uint64_t)(fm | 0x800000u);            /* 24 significant bits */
    if (e < -14) {                                        /* binary16 subnormal: units of 2^-24 */
        int sh = 23 - (e + 24);                           /* value / 2^-24 = sig * 2^(e+24-23) */
        uint64_t m = shift_rne(sig, sh);                  /* may round up to 0x400 = min normal */
        return (uint16_t)(sign | (uint16_t)m);
    }
    uint64_t m = shift_rne(sig, 13);                      /* 11 bits incl. the hidden one */
    int he = e + 15;
    if (m == 0x800u) { m = 0x400u; he++; }                /* mantissa overflow bumps the exponent */
    if (he >= 31) return (uint16_t)(sign | 0x7C00u);      /* overflow rounds to infinity */
    return (uint16_t)(sign | (uint16_t)(he << 10) | (uint16_t)(m & 0x3FFu));
}

/* ----------------------------------------------------------------------------- */
/* Element access and the reduction operator on raw bits.                          */
/* ----------------------------------------------------------------------------- */

static size_t elem_size(int dt) {
    switch (dt) {
    case ORC_F32: case ORC_I32: return 4;
    case ORC_F16: case ORC_BF16: return 2;
    default: return 0;
    }
}

static uint32_t load_bits(const void* p, size_t esz, size_t e) {
    const unsigned char* c = (const unsigned char*)p + e * esz;
    if (esz == 4) { uint32_t v; memcpy(&v, c, 4); return v; }
    uint16_t v; memcpy(&v, c, 2); return v;
}

static void store_bits(void* p, size_t esz, size_t e, uint32_t v) {
    unsigned char* c = (unsigned char*)p + e * esz;
    if (esz == 4) { memcpy(c, &v, 4); return; }
    uint16_t h = (uint16_t)v; memcpy(c, &h, 2);
}

static float to_f32(int dt, uint32_t v) {
    switch (dt) {
    case ORC_F32: return bits_to_f32(v);
    case ORC_F16: return orc_f16_to_f32((uint16_t)v);
    case ORC_BF16: return orc_bf16_to_f32((uint16_t)v);
    default: return (float)(int32_t)v;
    }
}

static uint32_t from_f32(int dt, float f) {
    switch (dt) {
    case ORC_F32: return f32_to_bits(f);
    case ORC_F16: return orc_f32_to_f16(f);
    default: return orc_f32_to_bf16(f);
    }
}

/* a = running partial (earlier ranks in ring order), b = the next rank's element. */
static uint32_t reduce_op(int dt, int op, uint32_t a, uint32_t b) {
    if (dt == ORC_I32) {
        int32_t sa = (int32_t)a, sb = (int32_t)b;
        switch (op) {
        case ORC_SUM: return a + b;                        /* wraps modulo 2^32 */
        case ORC_PROD: return a * b;
        case ORC_MIN: return (sb < sa) ? b : a;
        default: return (sb > sa) ? b : a;
        }
    }
    float fa = to_f32(dt, a), fb = to_f32(dt, b);
    switch (op) {
    case ORC_SUM: { volatile float r = fa + fb; return from_f32(dt, r); }
    case ORC_PROD: { volatile float r = fa * fb; return from_f32(dt, r); }
    case ORC_MIN: return (fb < fa) ? b : a;
    default: return (fb > fa) ? b : a;
    }
}

/* ---------------------------------------------------------------------------- */
/* Trees.                                                                          */
/* ---------------------------------------------------------------------------- */

/* Parent and children of `rank` in the binary tree over ranks 0..n-1: the tree hangs
 * from rank 0; a rank's lowest set bit `bit` fixes its level; its parent is the rank
 * with that bit cleared and the next one set (or just cleared when that is out of
 * range); its children are rank -/+ bit/2 (the right one shrunk until it is in range).
 * -1 marks a missing link. */
void orc_btree(int n, int rank, int* up, int* d0, int* d1) {
    int bit = 1;
    while (bit < n && !(bit & rank)) bit <<= 1;
    if (rank == 0) {
        *up = -1;
        *d0 = -1;
        *d1 = n > 1 ? bit >> 1 : -1;
        return;
    }
    int u = (rank ^ bit) | (bit << 1);
    if (u >= n) u = rank ^ bit;
    *up = u;
    int low = bit >> 1;
    *d0 = low ? rank - low : -1;
    int right = -1;
    while (low) {
        if (rank + low < n) { right = rank + low; break; }
        low >>= 1;
    }
    *d1 = right;
}

/* Tree `t` (0 or 1) of the double binary tree. */
void orc_dtree(int n, int rank, int t, int* up, int* d0, int* d1) {
    if (t == 0) { orc_btree(n, rank, up, d0, d1); return; }
    int u, a, b;
    if (n % 2 == 0) {                       /* mirror */
        orc_btree(n, n - 1 - rank, &u, &a, &b);
        *up = u < 0 ? -1 : n - 1 - u;
        *d0 = a < 0 ? -1 : n - 1 - a;
        *d1 = b < 0 ? -1 : n - 1 - b;
    } else {                                /* shift */
        orc_btree(n, (rank - 1 + n) % n, &u, &a, &b);
        *up = u < 0 ? -1 : (u + 1) % n;
        *d0 = a < 0 ? -1 : (a + 1) % n;
        *d1 = b < 0 ? -1 : (b + 1) % n;
    }
}

static int valid_dt_op(int dt, int op) {
    return elem_size(dt) != 0 && op >= ORC_SUM && op <= ORC_MAX;
}

/* ----------------------------------------------------------------------------- */
/* Reductions in ring order.                                                       */
/* ----------------------------------------------------------------------------- */

size_t orc_block_elems(size_t count, int n, size_t esz) {
    if (n < 1 || esz == 0 || esz > 16) return 0;
    size_t per = (count + (size_t)n - 1) / (size_t)n;     /* ceil(count / N) */
    size_t align = 16 / esz;
    return (per + align - 1) / align * align;              /* alignUp(., 16 / esz) */
}

/* Partial of element e of block b: ranks b+1, b+2, ..., b (mod N), one op each. */
static uint32_t ring_reduce(int dt, int op, int n, const void* const* x, size_t esz, size_t e, size_t b) {
    uint32_t acc = load_bits(x[(b + 1) % (size_t)n], esz, e);
    for (int k = 2; k <= n; k++) {
        uint32_t v = load_bits(x[(b + (size_t)k) % (size_t)n], esz, e);
        acc = reduce_op(dt, op, acc, v);
    }
    return acc;
}

typedef struct {
    int kind;                 /* 0 all-reduce, 1 reduce-scatter, 2 reduce-scatter + epilogue,
                                 3 reduce to root, 4 double-tree all-reduce */
    int dt, op, n, outdt;
    size_t count, recvcount, block;
    int root;
    float scale;
    const void* const* send;
    void* const* recv;
    size_t lo, hi;            /* element range [lo, hi) of the flat send index handled */
} job_t;

/* Partial of the subtree under `v` in tree t, element e. */
static uint32_t tree_reduce(int dt, int op, int n, const void* const* x, size_t esz, size_t e, int t, int v) {
    int up, d0, d1;
    orc_dtree(n, v, t, &up, &d0, &d1);
    uint32_t acc = load_bits(x[v], esz, e);
    if (d0 >= 0) acc = reduce_op(dt, op, acc, tree_reduce(dt, op, n, x, esz, e, t, d0));
    if (d1 >= 0) acc = reduce_op(dt, op, acc, tree_reduce(dt, op, n, x, esz, e, t, d1));
    return acc;
}

/* Root of tree t: the rank without a parent. */
static int tree_root(int n, int t) {
    for (int r = 0; r < n; r++) {
        int up, d0, d1;
        orc_dtree(n, r, t, &up, &d0, &d1);
        if (up < 0) return r;
    }
    return 0;
}

static void run_job(const job_t* j) {
    size_t esz = elem_size(j->dt);
    if (j->kind == 0) {
        for (size_t e = j->lo; e < j->hi; e++) {
            uint32_t acc = ring_reduce(j->dt, j->op, j->n, j->send, esz, e, e / j->block);
            for (int r = 0; r < j->n; r++) store_bits(j->recv[r], esz, e, acc);
        }
        return;
    }
    if (j->kind == 4) {
        /* first half (block = the split point) up tree 0, the rest up tree 1 */
        for (size_t e = j->lo; e < j->hi; e++) {
            const int t = e < j->block ? 0 : 1;
            const uint32_t acc = tree_reduce(j->dt, j->op, j->n, j->send, esz, e, t, tree_root(j->n, t));
            for (int r = 0; r < j->n; r++) store_bits(j->recv[r], esz, e, acc);
        }
        return;
    }
    if (j->kind == 3) {
        for (size_t e = j->lo; e < j->hi; e++)
            store_bits(j->recv[j->root], esz, e,
                       ring_reduce(j->dt, j->op, j->n, j->send, esz, e, (size_t)j->root));
        return;
    }
    /* reduce-scatter: flat index e = r * recvcount + t, block r lands in recv[r][t] */
    for (size_t e = j->lo; e < j->hi; e++) {
        size_t r = e / j->recvcount, t = e % j->recvcount;
        uint32_t acc = ring_reduce(j->dt, j->op, j->n, j->send, esz, e, r);
        if (j->kind == 1) {
            store_bits(j->recv[r], esz, t, acc);
        } else {
            volatile float y = to_f32(j->dt, acc) * j->scale;
            store_bits(j->recv[r], elem_size(j->outdt), t, from_f32(j->outdt, y));
        }
    }
}

static void* job_thread(void* p) { run_job((const job_t*)p); return NULL; }

#define ORC_MAX_THREADS 256

/* Split [0, total) into nthreads contiguous ranges.  Every element is still reduced
 * in the same ring order by exactly one thread, so the bits do not depend on it. */
static int run_split(job_t base, size_t total, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > ORC_MAX_THREADS) nthreads = ORC_MAX_THREADS;
    if ((size_t)nthreads > total) nthreads = total ? (int)total : 1;
    if (nthreads == 1) { base.lo = 0; base.hi = total; run_job(&base); return 0; }
    pthread_t th[ORC_MAX_THREADS];
    job_t jobs[ORC_MAX_THREADS];
    size_t per = (total + (size_t)nthreads - 1) / (size_t)nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = base;
        jobs[t].lo = (size_t)t * per < total ? (size_t)t * per : total;
        jobs[t].hi = jobs[t].lo + per < total ? jobs[t].lo + per : total;
        if (pthread_create(&th[t], NULL, job_thread, &jobs[t]) != 0) {
            run_job(&jobs[t]);                               /* fall back to this thread */
            th[t] = 0;
        } else {
            started++;
        }
    }
    for (int t = 0; t < nthreads; t++)
        if (th[t]) pthread_join(th[t], NULL);
    (void)started;
    return 0;
}

int orc_allreduce(int dt, int op, int n, size_t count, const void* const* send, void* const* recv,
                  int nthreads) {
    if (!valid_dt_op(dt, op) || n < 1) return -1;
    if (count == 0) return 0;
    if (!send || !recv) return -2;
    job_t j; memset(&j, 0, sizeof j);
    j.kind = 0; j.dt = dt; j.op = op; j.n = n; j.count = count;
    j.block = orc_block_elems(count, n, elem_size(dt));
    j.send = send; j.recv = recv;
    return run_split(j, count, nthreads);
}

int orc_reduce_scatter(int dt, int op, int n, size_t recvcount, const void* const* send,
                       void* const* recv, int nthreads) {
    if (!valid_dt_op(dt, op) || n < 1) return -1;
    if (recvcount == 0) return 0;
    if (!send || !recv) return -2;
    job_t j; memset(&j, 0, sizeof j);
    j.kind = 1; j.dt = dt; j.op = op; j.n = n; j.recvcount = recvcount;
    j.send = send; j.recv = recv;
    return run_split(j, recvcount * (size_t)n, nthreads);
}

/* Double-binary-tree all-reduce.  The split point between the two trees is
 * alignUp(ceil(count / 2), 16 / elemSize) elements. */
int orc_allreduce_tree(int dt, int op, int n, size_t count, const void* const* send, void* const* recv,
                       int nthreads) {
    if (!valid_dt_op(dt, op) || n < 1) return -1;
    if (count == 0) return 0;
    if (!send || !recv) return -2;
    job_t j; memset(&j, 0, sizeof j);
    j.kind = 4; j.dt = dt; j.op = op; j.n = n; j.count = count;
    j.block = orc_block_elems(count, 2, elem_size(dt));
    j.send = send; j.recv = recv;
    return run_split(j, count, nthreads);
}

/* Reduce to root: only recv[root] is written. */
int orc_reduce(int dt, int op, int n, size_t count, int root, const void* const* send,
               void* const* recv, int nthreads) {
    if (!valid_dt_op(dt, op) || n < 1 || root < 0 || root >= n) return -1;
    if (count == 0) return 0;
    if (!send || !recv || !recv[root]) return -2;
    job_t j; memset(&j, 0, sizeof j);
    j.kind = 3; j.dt = dt; j.op = op; j.n = n; j.count = count; j.root = root;
    j.send = send; j.recv = recv;
    return run_split(j, count, nthreads);
}

/* Reduce-scatter whose output element is (float)acc * scale, stored as outdt
 * (fp32, or the input type itself). */
int orc_reduce_scatter_scale(int dt, int op, int n, size_t recvcount, int outdt, float scale,
                             const void* const* send, void* const* recv, int nthreads) {
    if (!valid_dt_op(dt, op) || n < 1 || dt == ORC_I32) return -1;
    if (outdt != ORC_F32 && outdt != dt) return -1;
    if (recvcount == 0) return 0;
    if (!send || !recv) return -2;
    job_t j; memset(&j, 0, sizeof j);
    j.kind = 2; j.dt = dt; j.op = op; j.n = n; j.recvcount = recvcount;
    j.outdt = outdt; j.scale = scale; j.send = send; j.recv = recv;
    return run_split(j, recvcount * (size_t)n, nthreads);
}

/* ----------------------------------------------------------------------------- */
/* Data movement: byte copies.                                                     */
/* ----------------------------------------------------------------------------- */

int orc_allgather(size_t esz, int n, size_t sendcount, const void* const* send, void* const* recv) {
    if (n < 1 || esz == 0) return -1;
    if (sendcount == 0) return 0;
    size_t bytes = sendcount * esz;
    for (int r = 0; r < n; r++)
        for (int s = 0; s < n; s++)
            memmove((char*)recv[r] + (size_t)s * bytes, send[s], bytes);
    return 0;
}

int orc_broadcast(size_t esz, int n, size_t count, int root, const void* const* send, void* const* recv) {
    if (n < 1 || esz == 0 || root < 0 || root >= n) return -1;
    if (count == 0) return 0;
    for (int r = 0; r < n; r++) memmove(recv[r], send[root], count * esz);
    return 0;
}

int orc_gather(size_t esz, int n, size_t sendcount, int root, const void* const* send,
               void* const* recv) {
    if (n < 1 || esz == 0 || root < 0 || root >= n) return -1;
    if (sendcount == 0) return 0;
    size_t bytes = sendcount * esz;
    for (int s = 0; s < n; s++) memcpy((char*)recv[root] + (size_t)s * bytes, send[s], bytes);
    return 0;
}

int orc_scatter(size_t esz, int n, size_t recvcount, int root, const void* const* send,
                void* const* recv) {
    if (n < 1 || esz == 0 || root < 0 || root >= n) return -1;
    if (recvcount == 0) return 0;
    size_t bytes = recvcount * esz;
    for (int r = 0; r < n; r++) memcpy(recv[r], (const char*)send[root] + (size_t)r * bytes, bytes);
    return 0;
}

int orc_alltoall(size_t esz, int n, size_t count, const void* const* send, void* const* recv) {
    if (n < 1 || esz == 0) return -1;
    if (count == 0) return 0;
    size_t bytes = count * esz;
    for (int i = 0; i < n; i++)
        for (int j = 0; j < n; j++)
            memcpy((char*)recv[j] + (size_t)i * bytes, (const char*)send[i] + (size_t)j * bytes, bytes);
    return 0;
}

/* counts[i*n + j]: elements rank i sends to rank j; sdispls[i*n + j]: their offset in
 * send[i]; rdispls[j*n + i]: their offset in recv[j].  All in elements. */
int orc_alltoallv(size_t esz, int n, const int32_t* counts, const int32_t* sdispls,
                  const int32_t* rdispls, const void* const* send, void* const* recv) {
    if (n < 1 || esz == 0 || !counts || !sdispls || !rdispls) return -1;
    for (int i = 0; i < n; i++)
        for (int j = 0; j < n; j++) {
            int32_t c = counts[i * n + j], so = sdispls[i * n + j], ro = rdispls[j * n + i];
            if (c < 0 || so < 0 || ro < 0) return -1;
            if (c == 0) continue;
            memcpy((char*)recv[j] + (size_t)ro * esz, (const char*)send[i] + (size_t)so * esz,
                   (size_t)c * esz);
        }
    return 0;
}

/* Array forms of the conversions, for the unit tests that pin them. */
void orc_f32_to_type(int dt, size_t n, const float* in, void* out) {
    for (size_t i = 0; i < n; i++) store_bits(out, elem_size(dt), i, from_f32(dt, in[i]));
}

void orc_type_to_f32(int dt, size_t n, const void* in, float* out) {
    for (size_t i = 0; i < n; i++) out[i] = to_f32(dt, load_bits(in, elem_size(dt), i));
}
