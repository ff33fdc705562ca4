/*
 * orrery_oracle.c -- plain, slow CPU oracle of the Barnes-Hut monopole force
 * evaluation (stackless depth-first octree with escape indices).
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers. This file shares no code, header,
 * table or helper with the CUDA library in tree_traversal_gb300/, and neither
 * side includes or links the other.
 *
 * What it follows (the orrery documentation pages):
 *   [SOLVER]  "sycl_tree_solver.hpp" reference page: Detailed Description
 *             ("The mitigation", "What is not given up", "Where the tree comes
 *             from") and the TreeTraversal enumeration (kIndependent,
 *             kCoherent).
 *   [ADR29]   "ADR-0029: Mask the accepted cells rather than descending
 *             together": Decision and Consequences.
 *   [PERF]    "docs/performance/sycl_tree.md": "The machine and the device"
 *             table (Plummer sphere, softening 0.05, opening angle 0.5, leaf
 *             capacity 32, monopole only), "The divergence mitigation" (what
 *             a visit is), "Accuracy" (compensated fp64 direct sum).
 *   The force law a = m r / (r^2 + eps^2)^(3/2), the criterion "cell side /
 *   distance to centre of mass < theta" and the 21-bit-per-axis Morton cube
 *   come from the workload definition that accompanies the pages.
 *
 * Precision. The pages measure single precision. Every floating-point step
 * below is one binary32 operation rounded to nearest-even: +, -, *, /, fmaf
 * (one rounding) and sqrtf (correctly rounded, as IEEE 754 requires). The
 * force term is the law as written, m / (r2 sqrt(r2)), and nothing else: how
 * a kernel evaluates it is that kernel's choice. The file is compiled
 * with -ffp-contract=off so the compiler adds no fused operations.
 * Where the pages leave the arithmetic open, the reading taken is written at
 * the step; the same readings are listed in the design notes.
 *
 * Steps, in the order of one force evaluation:
 *   1 cube       oracle_cube
 *   2 keys       oracle_quantise, oracle_interleave, oracle_keys
 *   3 sort       oracle_sort
 *   4 tree       oracle_build
 *   5 moments    oracle_moments
 *   6-8 walk     oracle_walk (acceptance, leaf sums, force term)
 *   9 coherent   oracle_group_visits (union of the lanes' walks)
 *  10 output     oracle_bh_forces (whole evaluation, caller order)
 * Cross-checks: oracle_direct_f64 (compensated fp64 direct sum) and
 * oracle_bh_recursive (pointer tree, recursive walk, built separately).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_LEVELS 21 /* bits per axis in a key; deepest level */

/* ------------------------------------------------------------------------ */
/* Step 1: the bounding cube.                                               */
/* lo_a = min_i x_ia; the cube side is the largest per-axis extent          */
/* fl(max_i x_ia - lo_a); inv = fl(2^21 / side), or 0 when side is 0.       */
/* Reading: tight min corner, no padding, cube (not box).                   */
/* ------------------------------------------------------------------------ */
void oracle_cube(const float *pos, int64_t n, float lo[3], float *side, float *inv)
{
    float hi[3];
    for (int a = 0; a < 3; ++a) {
        lo[a] = 0.0f;
        hi[a] = 0.0f;
    }
    if (n > 0) {
        for (int a = 0; a < 3; ++a) {
            lo[a] = pos[a];
            hi[a] = pos[a];
        }
    }
    for (int64_t i = 1; i < n; ++i) {
        for (int a = 0; a < 3; ++a) {
            float x = pos[3 * i + a];
            if (x < lo[a]) lo[a] = x;
            if (x > hi[a]) hi[a] = x;
        }
    }
    float s = 0.0f;
    for (int a = 0; a < 3; ++a) {
        float ext = hi[a] - lo[a];
        if (ext > s) s = ext;
    }
    *side = s;
    *inv = (s > 0.0f) ? (2097152.0f / s) : 0.0f;
}

/* ------------------------------------------------------------------------ */
/* Step 2: quantise each axis to 21 bits and interleave.                    */
/* q = min(floor(fl(fl(x - lo) * inv)), 2^21 - 1).                          */
/* The key holds, for bit b = 20 (top) .. 0, the triple (x_b, y_b, z_b),     */
/* x highest: so the top triple is the level-1 octant, x the octant's       */
/* high bit. Reading: x is the high bit; children in ascending octant.      */
/* ------------------------------------------------------------------------ */
uint32_t oracle_quantise(float x, float lo, float inv)
{
    float t = (x - lo) * inv;
    if (!(t >= 0.0f)) t = 0.0f; /* x >= lo always for finite input */
    if (t >= 2097151.0f) return 2097151u;
    return (uint32_t)floorf(t);
}

uint64_t oracle_interleave(uint32_t qx, uint32_t qy, uint32_t qz)
{
    uint64_t key = 0;
    for (int b = 0; b < ORACLE_LEVELS; ++b) {
        uint64_t xb = (qx >> b) & 1u;
        uint64_t yb = (qy >> b) & 1u;
        uint64_t zb = (qz >> b) & 1u;
        key |= xb << (3 * b + 2);
        key |= yb << (3 * b + 1);
        key |= zb << (3 * b);
    }
    return key;
}

void oracle_keys(const float *pos, int64_t n, const float lo[3], float inv, uint64_t *keys)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t qx = oracle_quantise(pos[3 * i + 0], lo[0], inv);
        uint32_t qy = oracle_quantise(pos[3 * i + 1], lo[1], inv);
        uint32_t qz = oracle_quantise(pos[3 * i + 2], lo[2], inv);
        keys[i] = oracle_interleave(qx, qy, qz);
    }
}

/* ------------------------------------------------------------------------ */
/* Step 3: sort the (key, original index) pairs lexicographically.         */
/* Equal keys keep their original order (a stable sort by key).             */
/* ------------------------------------------------------------------------ */
typedef struct {
    uint64_t key;
    uint32_t index;
} key_index;

static int cmp_key_index(const void *pa, const void *pb)
{
    const key_index *a = (const key_index *)pa;
    const key_index *b = (const key_index *)pb;
    if (a->key != b->key) return (a->key < b->key) ? -1 : 1;
    if (a->index != b->index) return (a->index < b->index) ? -1 : 1;
    return 0;
}

int oracle_sort(const uint64_t *keys, int64_t n, uint32_t *perm, uint64_t *sorted_keys)
{
    key_index *pairs = (key_index *)malloc((size_t)(n > 0 ? n : 1) * sizeof(key_index));
    if (!pairs) return -1;
    for (int64_t i = 0; i < n; ++i) {
        pairs[i].key = keys[i];
        pairs[i].index = (uint32_t)i;
    }
    qsort(pairs, (size_t)n, sizeof(key_index), cmp_key_index);
    for (int64_t k = 0; k < n; ++k) {
        perm[k] = pairs[k].index;
        sorted_keys[k] = pairs[k].key;
    }
    free(pairs);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 4: the octree, built recursively over sorted ranges.                */
/* A node is a leaf iff count <= leaf_cap or its level is 21. Otherwise it  */
/* gets one child per non-empty octant, in ascending octant order (a node   */
/* with a single child keeps it). Nodes are written in depth-first          */
/* preorder; escape(k) is the index of the first node after k's subtree.    */
/* Node record: {escape, first, count, level} (four int32).                 */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint64_t *keys;
    int32_t leaf_cap;
    int32_t *nodes;
    int64_t max_nodes;
    int64_t num_nodes;
    int overflow;
} build_state;

static int octant_at(uint64_t key, int parent_level)
{
    /* the octant of a key inside a cell of level parent_level */
    return (int)((key >> (3 * (ORACLE_LEVELS - 1 - parent_level))) & 7u);
}

static void build_node(build_state *st, int64_t first, int64_t count, int level)
{
    int64_t k = st->num_nodes;
    st->num_nodes += 1;
    if (k >= st->max_nodes) {
        st->overflow = 1;
        return;
    }
    st->nodes[4 * k + 1] = (int32_t)first;
    st->nodes[4 * k + 2] = (int32_t)count;
    st->nodes[4 * k + 3] = level;
    int is_leaf = (count <= st->leaf_cap) || (level == ORACLE_LEVELS);
    if (!is_leaf) {
        int64_t j = first;
        int64_t end = first + count;
        for (int o = 0; o < 8; ++o) {
            int64_t start = j;
            while (j < end && octant_at(st->keys[j], level) == o) ++j;
            if (j > start) build_node(st, start, j - start, level + 1);
        }
    }
    if (k < st->max_nodes) st->nodes[4 * k + 0] = (int32_t)st->num_nodes;
}

int64_t oracle_build(const uint64_t *sorted_keys, int64_t n, int32_t leaf_cap,
                     int32_t *nodes, int64_t max_nodes)
{
    build_state st;
    st.keys = sorted_keys;
    st.leaf_cap = leaf_cap;
    st.nodes = nodes;
    st.max_nodes = max_nodes;
    st.num_nodes = 0;
    st.overflow = 0;
    if (n > 0) build_node(&st, 0, n, 0);
    if (st.overflow) return -1;
    return st.num_nodes;
}

static int node_is_leaf(const int32_t *node, int32_t leaf_cap)
{
    return node[2] <= leaf_cap || node[3] == ORACLE_LEVELS;
}

/* ------------------------------------------------------------------------ */
/* Step 5: monopole moments, upward.                                        */
/* Leaf: M = sum m_j and S_a = sum m_j x_ja over its particles in sorted    */
/*       order, S accumulated as fmaf(m_j, x_ja, S_a).                      */
/* Internal: M and S_a are the sums of the children's, in child order.      */
/* CoM_a = fl(S_a / M) when M > 0, else 0.                                  */
/* Output per node: {CoM_x, CoM_y, CoM_z, M}.                               */
/* Reading: fp32, sequential, fixed order, so that acceptance decisions are  */
/* reproducible bit for bit.                                                */
/* ps: sorted particles, 4 floats each {x, y, z, m}.                        */
/* ------------------------------------------------------------------------ */
static int64_t moments_node(const float *ps, const int32_t *nodes, int32_t leaf_cap,
                            int64_t k, float *S, float *cm)
{
    const int32_t *node = nodes + 4 * k;
    float M = 0.0f, sx = 0.0f, sy = 0.0f, sz = 0.0f;
    if (node_is_leaf(node, leaf_cap)) {
        for (int64_t j = node[1]; j < (int64_t)node[1] + node[2]; ++j) {
            float m = ps[4 * j + 3];
            M = M + m;
            sx = fmaf(m, ps[4 * j + 0], sx);
            sy = fmaf(m, ps[4 * j + 1], sy);
            sz = fmaf(m, ps[4 * j + 2], sz);
        }
    } else {
        int64_t c = k + 1;
        while (c < node[0]) {
            moments_node(ps, nodes, leaf_cap, c, S, cm);
            M = M + S[4 * c + 3];
            sx = sx + S[4 * c + 0];
            sy = sy + S[4 * c + 1];
            sz = sz + S[4 * c + 2];
            c = nodes[4 * c + 0];
        }
    }
    S[4 * k + 0] = sx;
    S[4 * k + 1] = sy;
    S[4 * k + 2] = sz;
    S[4 * k + 3] = M;
    cm[4 * k + 0] = (M > 0.0f) ? sx / M : 0.0f;
    cm[4 * k + 1] = (M > 0.0f) ? sy / M : 0.0f;
    cm[4 * k + 2] = (M > 0.0f) ? sz / M : 0.0f;
    cm[4 * k + 3] = M;
    return nodes[4 * k + 0];
}

int oracle_moments(const float *ps, const int32_t *nodes, int64_t num_nodes, int32_t leaf_cap,
                   float *cm)
{
    if (num_nodes <= 0) return 0;
    float *S = (float *)malloc((size_t)num_nodes * 4 * sizeof(float));
    if (!S) return -1;
    moments_node(ps, nodes, leaf_cap, 0, S, cm);
    free(S);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Steps 6-8: the walk of one target.                                       */
/*                                                                          */
/* Acceptance at node k of level L for target x_i (criterion "cell side /   */
/* distance to CoM < theta", squared):                                      */
/*   dx_a = fl(CoM_a - x_ia)                                                */
/*   d2   = fmaf(dz, dz, fmaf(dy, dy, fl(dx * dx)))                         */
/*   s2_L = fl(side * side) * 2^(-2L)   (the geometric cell side squared)   */
/*   accept iff s2_L < fl(fl(theta * theta) * d2)                           */
/* Reading: the test applies to every node, root and leaves included; the  */
/* comparison is strict; a target inside an accepted cell gets no special   */
/* case. d2 = 0 is never accepted; theta = 0 never accepts.                 */
/*                                                                          */
/* Term for a source (x_j, m_j): the softened law of the workload           */
/* definition, a = m r / (r^2 + eps^2)^(3/2), G = 1, written out plainly:   */
/*   r2 = fl(d2 + eps2), eps2 = fl(eps * eps)                               */
/*   f  = fl(m_j / fl(r2 * sqrtf(r2)))      (m_j r2^(-3/2))                 */
/*   a_ia = fmaf(f, dx_a, a_ia), in walk order                              */
/* Cell terms use (M, CoM) with the d2 of the acceptance test.              */
/*                                                                          */
/* The walk: k = 0; while k < num_nodes: visits++; accepted -> cell term,   */
/* pc++, k = escape; else a leaf -> every particle j of the leaf in sorted   */
/* order, j != i, particle term, pp++, then k = escape; else k = k + 1.     */
/* A visit is one node at which the acceptance test runs.                    */
/* ------------------------------------------------------------------------ */
typedef struct {
    const float *ps;      /* sorted particles {x, y, z, m} */
    const int32_t *nodes; /* {escape, first, count, level} */
    const float *cm;      /* {CoM_x, CoM_y, CoM_z, M} */
    int64_t num_nodes;
    int32_t leaf_cap;
    float side;
    float theta;
    float eps;
} walk_tree;

static float cell_side_sq(float side, int level)
{
    return ldexpf(side * side, -2 * level);
}

static void add_term(const float xi[3], float xj, float yj, float zj, float m, float eps2,
                     float acc[3])
{
    float dx = xj - xi[0];
    float dy = yj - xi[1];
    float dz = zj - xi[2];
    float d2 = fmaf(dz, dz, fmaf(dy, dy, dx * dx));
    float r2 = d2 + eps2;
    float f = m / (r2 * sqrtf(r2));
    acc[0] = fmaf(f, dx, acc[0]);
    acc[1] = fmaf(f, dy, acc[1]);
    acc[2] = fmaf(f, dz, acc[2]);
}

static int accept_cell(const float xi[3], const float *cm, float side, int level, float theta2)
{
    float dx = cm[0] - xi[0];
    float dy = cm[1] - xi[1];
    float dz = cm[2] - xi[2];
    float d2 = fmaf(dz, dz, fmaf(dy, dy, dx * dx));
    return cell_side_sq(side, level) < theta2 * d2;
}

static void walk_one(const walk_tree *t, int64_t i, float acc[3], uint32_t *pc, uint32_t *pp,
                     uint32_t *visits, uint8_t *visited)
{
    const float xi[3] = {t->ps[4 * i + 0], t->ps[4 * i + 1], t->ps[4 * i + 2]};
    const float theta2 = t->theta * t->theta;
    const float eps2 = t->eps * t->eps;
    acc[0] = acc[1] = acc[2] = 0.0f;
    *pc = *pp = *visits = 0;
    int64_t k = 0;
    while (k < t->num_nodes) {
        const int32_t *node = t->nodes + 4 * k;
        const float *c = t->cm + 4 * k;
        *visits += 1;
        if (visited) visited[k] = 1;
        if (accept_cell(xi, c, t->side, node[3], theta2)) {
            add_term(xi, c[0], c[1], c[2], c[3], eps2, acc);
            *pc += 1;
            k = node[0];
        } else if (node_is_leaf(node, t->leaf_cap)) {
            for (int64_t j = node[1]; j < (int64_t)node[1] + node[2]; ++j) {
                if (j == i) continue;
                const float *p = t->ps + 4 * j;
                add_term(xi, p[0], p[1], p[2], p[3], eps2, acc);
                *pp += 1;
            }
            k = node[0];
        } else {
            k = k + 1;
        }
    }
}

/* Worker pool over targets: contiguous slices, no shared writes. */
typedef struct {
    const walk_tree *tree;
    const int64_t *targets; /* sorted indices, or NULL for 0..count-1 */
    int64_t begin, end;
    float *acc;
    uint32_t *pc, *pp, *visits;
} walk_slice;

static void *walk_worker(void *arg)
{
    walk_slice *s = (walk_slice *)arg;
    for (int64_t q = s->begin; q < s->end; ++q) {
        int64_t i = s->targets ? s->targets[q] : q;
        uint32_t a, b, v;
        walk_one(s->tree, i, s->acc + 3 * q, &a, &b, &v, NULL);
        if (s->pc) s->pc[q] = a;
        if (s->pp) s->pp[q] = b;
        if (s->visits) s->visits[q] = v;
    }
    return NULL;
}

/* Walks the targets (sorted indices; NULL = all n_targets from 0) over the
 * tree. Outputs are per target in the order given. threads >= 1. */
int oracle_walk(const float *ps, const int32_t *nodes, const float *cm, int64_t num_nodes,
                int32_t leaf_cap, float side, float theta, float eps, const int64_t *targets,
                int64_t n_targets, float *acc, uint32_t *pc, uint32_t *pp, uint32_t *visits,
                int threads)
{
    walk_tree t = {ps, nodes, cm, num_nodes, leaf_cap, side, theta, eps};
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n_targets < threads) threads = (int)(n_targets > 0 ? n_targets : 1);
    pthread_t tid[256];
    walk_slice sl[256];
    for (int w = 0; w < threads; ++w) {
        sl[w].tree = &t;
        sl[w].targets = targets;
        sl[w].begin = n_targets * w / threads;
        sl[w].end = n_targets * (w + 1) / threads;
        sl[w].acc = acc;
        sl[w].pc = pc;
        sl[w].pp = pp;
        sl[w].visits = visits;
    }
    if (threads == 1) {
        walk_worker(&sl[0]);
        return 0;
    }
    for (int w = 0; w < threads; ++w)
        if (pthread_create(&tid[w], NULL, walk_worker, &sl[w]) != 0) return -1;
    for (int w = 0; w < threads; ++w) pthread_join(tid[w], NULL);
    return 0;
}

/* Marks (0/1) every node the walk of sorted target i visits. */
void oracle_walk_marks(const float *ps, const int32_t *nodes, const float *cm, int64_t num_nodes,
                       int32_t leaf_cap, float side, float theta, float eps, int64_t i,
                       uint8_t *visited)
{
    walk_tree t = {ps, nodes, cm, num_nodes, leaf_cap, side, theta, eps};
    float acc[3];
    uint32_t a, b, v;
    memset(visited, 0, (size_t)num_nodes);
    walk_one(&t, i, acc, &a, &b, &v, visited);
}

/* ------------------------------------------------------------------------ */
/* Step 9: the coherent walk's visit count ([ADR29] Decision).              */
/* A group of `width` consecutive sorted targets shares one node index and  */
/* advances to the smallest index any lane still wants, so the group visits */
/* exactly the union of its lanes' own walks, and each lane's visit counter */
/* is the size of that union. Group g holds targets g*width .. (g+1)*width-1 */
/* (the last group is truncated at n). Output: union size per group.        */
/* ------------------------------------------------------------------------ */
int oracle_group_visits(const float *ps, const int32_t *nodes, const float *cm, int64_t num_nodes,
                        int32_t leaf_cap, float side, float theta, float eps, int64_t n,
                        int32_t width, const int64_t *groups, int64_t n_groups,
                        uint32_t *union_size)
{
    walk_tree t = {ps, nodes, cm, num_nodes, leaf_cap, side, theta, eps};
    uint8_t *mark = (uint8_t *)malloc((size_t)(num_nodes > 0 ? num_nodes : 1));
    if (!mark) return -1;
    for (int64_t q = 0; q < n_groups; ++q) {
        int64_t g = groups ? groups[q] : q;
        memset(mark, 0, (size_t)num_nodes);
        for (int64_t i = g * width; i < (g + 1) * width && i < n; ++i) {
            float acc[3];
            uint32_t a, b, v;
            walk_one(&t, i, acc, &a, &b, &v, mark);
        }
        uint32_t cnt = 0;
        for (int64_t k = 0; k < num_nodes; ++k) cnt += mark[k];
        union_size[q] = cnt;
    }
    free(mark);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The rejected alternative, for comparison ([ADR29] Alternatives considered,*/
/* "Descend wherever any lane must, and let the accepting lanes descend      */
/* too"). A group of `width` consecutive sorted targets walks one node       */
/* index. At node k every target of the group takes the criterion; if all   */
/* accept, each adds the cell term and the group jumps to escape(k); else   */
/* if k is a leaf, each adds the terms of all the leaf's particles but its   */
/* own and the group jumps to escape(k); else the group descends to k + 1,  */
/* the would-be acceptors with it. Each target's sum now depends on which   */
/* targets share its group. Counters are per target as in the walk; visits */
/* are the group's steps. Outputs in sorted order.                           */
/* ------------------------------------------------------------------------ */
int oracle_descend_together(const float *ps, const int32_t *nodes, const float *cm,
                            int64_t num_nodes, int32_t leaf_cap, float side, float theta,
                            float eps, int64_t n, int32_t width, float *acc, uint32_t *pc,
                            uint32_t *pp, uint32_t *visits)
{
    const float theta2 = theta * theta;
    const float eps2 = eps * eps;
    for (int64_t g = 0; g * width < n; ++g) {
        const int64_t lo = g * width;
        const int64_t hi = (lo + width < n) ? lo + width : n;
        for (int64_t i = lo; i < hi; ++i) {
            acc[3 * i] = acc[3 * i + 1] = acc[3 * i + 2] = 0.0f;
            pc[i] = pp[i] = visits[i] = 0;
        }
        int64_t k = 0;
        while (k < num_nodes) {
            const int32_t *node = nodes + 4 * k;
            const float *c = cm + 4 * k;
            int all_accept = 1;
            for (int64_t i = lo; i < hi; ++i) {
                const float xi[3] = {ps[4 * i], ps[4 * i + 1], ps[4 * i + 2]};
                visits[i] += 1;
                if (!accept_cell(xi, c, side, node[3], theta2)) all_accept = 0;
            }
            if (all_accept) {
                for (int64_t i = lo; i < hi; ++i) {
                    const float xi[3] = {ps[4 * i], ps[4 * i + 1], ps[4 * i + 2]};
                    add_term(xi, c[0], c[1], c[2], c[3], eps2, acc + 3 * i);
                    pc[i] += 1;
                }
                k = node[0];
            } else if (node_is_leaf(node, leaf_cap)) {
                for (int64_t i = lo; i < hi; ++i) {
                    const float xi[3] = {ps[4 * i], ps[4 * i + 1], ps[4 * i + 2]};
                    for (int64_t j = node[1]; j < (int64_t)node[1] + node[2]; ++j) {
                        if (j == i) continue;
                        add_term(xi, ps[4 * j], ps[4 * j + 1], ps[4 * j + 2], ps[4 * j + 3], eps2,
                                 acc + 3 * i);
                        pp[i] += 1;
                    }
                }
                k = node[0];
            } else {
                k = k + 1;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 10: one whole force evaluation, outputs in the caller's order.      */
/* Gathers the particles into tree order and scatters the results back      */
/* ([SOLVER] "Where the tree comes from").                                  */
/* interactions: 2 per particle {particle-cell, particle-particle}.          */
/* visits_ind: the particle's own walk. visits_coh (may be NULL): the union */
/* of its 32-wide group in sorted order.                                    */
/* Returns the node count, or a negative value on failure.                  */
/* ------------------------------------------------------------------------ */
int64_t oracle_bh_forces(const float *pos, const float *mass, int64_t n, float theta, float eps,
                         int32_t leaf_cap, float *acc, uint32_t *interactions,
                         uint32_t *visits_ind, uint32_t *visits_coh, int threads)
{
    if (n <= 0) return 0;
    float lo[3], side, inv;
    oracle_cube(pos, n, lo, &side, &inv);
    uint64_t *keys = (uint64_t *)malloc((size_t)n * sizeof(uint64_t));
    uint64_t *sorted = (uint64_t *)malloc((size_t)n * sizeof(uint64_t));
    uint32_t *perm = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    float *ps = (float *)malloc((size_t)n * 4 * sizeof(float));
    int64_t max_nodes = 22 * n + 1;
    int32_t *nodes = (int32_t *)malloc((size_t)max_nodes * 4 * sizeof(int32_t));
    float *acc_s = (float *)malloc((size_t)n * 3 * sizeof(float));
    uint32_t *pc = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    uint32_t *pp = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    uint32_t *vis = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    float *cm = NULL;
    int64_t num_nodes = -1;
    if (!keys || !sorted || !perm || !ps || !nodes || !acc_s || !pc || !pp || !vis) goto done;
    oracle_keys(pos, n, lo, inv, keys);
    if (oracle_sort(keys, n, perm, sorted) != 0) goto done;
    for (int64_t k = 0; k < n; ++k) {
        uint32_t i = perm[k];
        ps[4 * k + 0] = pos[3 * i + 0];
        ps[4 * k + 1] = pos[3 * i + 1];
        ps[4 * k + 2] = pos[3 * i + 2];
        ps[4 * k + 3] = mass[i];
    }
    num_nodes = oracle_build(sorted, n, leaf_cap, nodes, max_nodes);
    if (num_nodes < 0) goto done;
    cm = (float *)malloc((size_t)num_nodes * 4 * sizeof(float));
    if (!cm || oracle_moments(ps, nodes, num_nodes, leaf_cap, cm) != 0) {
        num_nodes = -1;
        goto done;
    }
    if (oracle_walk(ps, nodes, cm, num_nodes, leaf_cap, side, theta, eps, NULL, n, acc_s, pc, pp,
                    vis, threads) != 0) {
        num_nodes = -1;
        goto done;
    }
    for (int64_t k = 0; k < n; ++k) {
        uint32_t i = perm[k];
        acc[3 * i + 0] = acc_s[3 * k + 0];
        acc[3 * i + 1] = acc_s[3 * k + 1];
        acc[3 * i + 2] = acc_s[3 * k + 2];
        if (interactions) {
            interactions[2 * i + 0] = pc[k];
            interactions[2 * i + 1] = pp[k];
        }
        if (visits_ind) visits_ind[i] = vis[k];
    }
    if (visits_coh) {
        int64_t ng = (n + 31) / 32;
        uint32_t *u = (uint32_t *)malloc((size_t)ng * sizeof(uint32_t));
        if (!u || oracle_group_visits(ps, nodes, cm, num_nodes, leaf_cap, side, theta, eps, n, 32,
                                      NULL, ng, u) != 0) {
            free(u);
            num_nodes = -1;
            goto done;
        }
        for (int64_t k = 0; k < n; ++k) visits_coh[perm[k]] = u[k / 32];
        free(u);
    }
done:
    free(keys);
    free(sorted);
    free(perm);
    free(ps);
    free(nodes);
    free(acc_s);
    free(pc);
    free(pp);
    free(vis);
    free(cm);
    return num_nodes;
}

/* ------------------------------------------------------------------------ */
/* Cross-check 1: direct summation in fp64 with Neumaier compensation, the  */
/* stand-in for the pages' compensated double-precision reference kernel    */
/* ([PERF] Accuracy). Same softened law, every pair j != i.                  */
/* targets: original indices (NULL = 0..n_targets-1). acc: 3 doubles each.  */
/* ------------------------------------------------------------------------ */
typedef struct {
    const float *pos, *mass;
    int64_t n;
    double eps2;
    const int64_t *targets;
    int64_t begin, end;
    double *acc;
} direct_slice;

static void neumaier_add(double *s, double *c, double v)
{
    double t = *s + v;
    if (fabs(*s) >= fabs(v))
        *c += (*s - t) + v;
    else
        *c += (v - t) + *s;
    *s = t;
}

static void *direct_worker(void *arg)
{
    direct_slice *d = (direct_slice *)arg;
    for (int64_t q = d->begin; q < d->end; ++q) {
        int64_t i = d->targets ? d->targets[q] : q;
        double xi = d->pos[3 * i], yi = d->pos[3 * i + 1], zi = d->pos[3 * i + 2];
        double s[3] = {0, 0, 0}, c[3] = {0, 0, 0};
        for (int64_t j = 0; j < d->n; ++j) {
            if (j == i) continue;
            double dx = (double)d->pos[3 * j] - xi;
            double dy = (double)d->pos[3 * j + 1] - yi;
            double dz = (double)d->pos[3 * j + 2] - zi;
            double r2 = dx * dx + dy * dy + dz * dz + d->eps2;
            double f = (double)d->mass[j] / (r2 * sqrt(r2));
            neumaier_add(&s[0], &c[0], f * dx);
            neumaier_add(&s[1], &c[1], f * dy);
            neumaier_add(&s[2], &c[2], f * dz);
        }
        for (int a = 0; a < 3; ++a) d->acc[3 * q + a] = s[a] + c[a];
    }
    return NULL;
}

int oracle_direct_f64(const float *pos, const float *mass, int64_t n, double eps,
                      const int64_t *targets, int64_t n_targets, double *acc, int threads)
{
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n_targets < threads) threads = (int)(n_targets > 0 ? n_targets : 1);
    pthread_t tid[256];
    direct_slice sl[256];
    for (int w = 0; w < threads; ++w) {
        sl[w].pos = pos;
        sl[w].mass = mass;
        sl[w].n = n;
        sl[w].eps2 = eps * eps;
        sl[w].targets = targets;
        sl[w].begin = n_targets * w / threads;
        sl[w].end = n_targets * (w + 1) / threads;
        sl[w].acc = acc;
    }
    if (threads == 1) {
        direct_worker(&sl[0]);
        return 0;
    }
    for (int w = 0; w < threads; ++w)
        if (pthread_create(&tid[w], NULL, direct_worker, &sl[w]) != 0) return -1;
    for (int w = 0; w < threads; ++w) pthread_join(tid[w], NULL);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The scale of a target's sum: S_i = sum over j != i of the magnitudes of   */
/* its terms, m_j |x_j - x_i| / (|x_j - x_i|^2 + eps^2)^(3/2), in fp64.      */
/* A sum of terms that nearly cancel (a target at the centre of a symmetric */
/* distribution, or close unsoftened pairs) has |a_i| far below S_i; every */
/* per-term rounding error is relative to its term, so the deviation of two */
/* correct fp32 evaluations is bounded by a multiple of S_i, not of |a_i|.  */
/* targets: original indices (NULL = 0..n_targets-1).                       */
/* ------------------------------------------------------------------------ */
static void *magnitude_worker(void *arg)
{
    direct_slice *d = (direct_slice *)arg;
    for (int64_t q = d->begin; q < d->end; ++q) {
        int64_t i = d->targets ? d->targets[q] : q;
        double xi = d->pos[3 * i], yi = d->pos[3 * i + 1], zi = d->pos[3 * i + 2];
        double s = 0.0;
        for (int64_t j = 0; j < d->n; ++j) {
            if (j == i) continue;
            double dx = (double)d->pos[3 * j] - xi;
            double dy = (double)d->pos[3 * j + 1] - yi;
            double dz = (double)d->pos[3 * j + 2] - zi;
            double d2 = dx * dx + dy * dy + dz * dz;
            double r2 = d2 + d->eps2;
            if (r2 > 0.0) s += fabs((double)d->mass[j]) * sqrt(d2) / (r2 * sqrt(r2));
        }
        d->acc[q] = s;
    }
    return NULL;
}

int oracle_term_magnitude_f64(const float *pos, const float *mass, int64_t n, double eps,
                              const int64_t *targets, int64_t n_targets, double *out,
                              int threads)
{
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n_targets < threads) threads = (int)(n_targets > 0 ? n_targets : 1);
    pthread_t tid[256];
    direct_slice sl[256];
    for (int w = 0; w < threads; ++w) {
        sl[w].pos = pos;
        sl[w].mass = mass;
        sl[w].n = n;
        sl[w].eps2 = eps * eps;
        sl[w].targets = targets;
        sl[w].begin = n_targets * w / threads;
        sl[w].end = n_targets * (w + 1) / threads;
        sl[w].acc = out;
    }
    if (threads == 1) {
        magnitude_worker(&sl[0]);
        return 0;
    }
    for (int w = 0; w < threads; ++w)
        if (pthread_create(&tid[w], NULL, magnitude_worker, &sl[w]) != 0) return -1;
    for (int w = 0; w < threads; ++w) pthread_join(tid[w], NULL);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Direct summation in binary32 with the walk's own particle term, j        */
/* ascending in caller order, j != i: the GPU direct kernel's definition    */
/* (the pages' Phase 9 solver, [PERF] "Against the two solvers it has to    */
/* beat"). targets: original indices (NULL = 0..n_targets-1).               */
/* ------------------------------------------------------------------------ */
typedef struct {
    const float *pos, *mass;
    int64_t n;
    float eps2;
    const int64_t *targets;
    int64_t begin, end;
    float *acc;
} direct32_slice;

static void *direct32_worker(void *arg)
{
    direct32_slice *d = (direct32_slice *)arg;
    for (int64_t q = d->begin; q < d->end; ++q) {
        int64_t i = d->targets ? d->targets[q] : q;
        const float xi[3] = {d->pos[3 * i], d->pos[3 * i + 1], d->pos[3 * i + 2]};
        float a[3] = {0.0f, 0.0f, 0.0f};
        for (int64_t j = 0; j < d->n; ++j) {
            if (j == i) continue;
            add_term(xi, d->pos[3 * j], d->pos[3 * j + 1], d->pos[3 * j + 2], d->mass[j], d->eps2, a);
        }
        for (int c = 0; c < 3; ++c) d->acc[3 * q + c] = a[c];
    }
    return NULL;
}

int oracle_direct_f32(const float *pos, const float *mass, int64_t n, float eps,
                      const int64_t *targets, int64_t n_targets, float *acc, int threads)
{
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n_targets < threads) threads = (int)(n_targets > 0 ? n_targets : 1);
    pthread_t tid[256];
    direct32_slice sl[256];
    for (int w = 0; w < threads; ++w) {
        sl[w].pos = pos;
        sl[w].mass = mass;
        sl[w].n = n;
        sl[w].eps2 = eps * eps;
        sl[w].targets = targets;
        sl[w].begin = n_targets * w / threads;
        sl[w].end = n_targets * (w + 1) / threads;
        sl[w].acc = acc;
    }
    if (threads == 1) {
        direct32_worker(&sl[0]);
        return 0;
    }
    for (int w = 0; w < threads; ++w)
        if (pthread_create(&tid[w], NULL, direct32_worker, &sl[w]) != 0) return -1;
    for (int w = 0; w < threads; ++w) pthread_join(tid[w], NULL);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Cross-check 2: a pointer octree built and walked recursively.            */
/* Built on its own from the sorted keys (an explicit child array per cell, */
/* no escape indices), moments by recursion, and a recursive walk that       */
/* opens children in octant order. Same criterion and term, so it must equal */
/* the escape-index walk bit for bit: that pins the escape indices and the  */
/* depth-first layout.                                                      */
/* ------------------------------------------------------------------------ */
typedef struct pnode {
    int64_t first, count;
    int level;
    int nchild;
    struct pnode *child[8];
    float M, sx, sy, sz, cx, cy, cz;
} pnode;

static pnode *pbuild(const uint64_t *keys, const float *ps, int64_t first, int64_t count,
                     int level, int32_t leaf_cap)
{
    pnode *p = (pnode *)calloc(1, sizeof(pnode));
    if (!p) return NULL;
    p->first = first;
    p->count = count;
    p->level = level;
    if (count > leaf_cap && level < ORACLE_LEVELS) {
        for (int o = 0; o < 8; ++o) {
            int64_t a = -1, b = -1;
            for (int64_t j = first; j < first + count; ++j) {
                if (octant_at(keys[j], level) == o) {
                    if (a < 0) a = j;
                    b = j;
                }
            }
            if (a >= 0) p->child[p->nchild++] = pbuild(keys, ps, a, b - a + 1, level + 1, leaf_cap);
        }
        for (int c = 0; c < p->nchild; ++c) {
            pnode *ch = p->child[c];
            p->M = p->M + ch->M;
            p->sx = p->sx + ch->sx;
            p->sy = p->sy + ch->sy;
            p->sz = p->sz + ch->sz;
        }
    } else {
        for (int64_t j = first; j < first + count; ++j) {
            float m = ps[4 * j + 3];
            p->M = p->M + m;
            p->sx = fmaf(m, ps[4 * j + 0], p->sx);
            p->sy = fmaf(m, ps[4 * j + 1], p->sy);
            p->sz = fmaf(m, ps[4 * j + 2], p->sz);
        }
    }
    p->cx = p->M > 0.0f ? p->sx / p->M : 0.0f;
    p->cy = p->M > 0.0f ? p->sy / p->M : 0.0f;
    p->cz = p->M > 0.0f ? p->sz / p->M : 0.0f;
    return p;
}

static void pfree(pnode *p)
{
    if (!p) return;
    for (int c = 0; c < p->nchild; ++c) pfree(p->child[c]);
    free(p);
}

static void pwalk(const pnode *p, const float *ps, int64_t i, const float xi[3], float side,
                  float theta2, float eps2, float acc[3], uint32_t cnt[3])
{
    cnt[2] += 1;
    float cmv[3] = {p->cx, p->cy, p->cz};
    if (accept_cell(xi, cmv, side, p->level, theta2)) {
        add_term(xi, p->cx, p->cy, p->cz, p->M, eps2, acc);
        cnt[0] += 1;
    } else if (p->nchild == 0) {
        for (int64_t j = p->first; j < p->first + p->count; ++j) {
            if (j == i) continue;
            add_term(xi, ps[4 * j], ps[4 * j + 1], ps[4 * j + 2], ps[4 * j + 3], eps2, acc);
            cnt[1] += 1;
        }
    } else {
        for (int c = 0; c < p->nchild; ++c)
            pwalk(p->child[c], ps, i, xi, side, theta2, eps2, acc, cnt);
    }
}

/* Whole evaluation through the pointer tree; outputs in sorted order
 * (acc 3 floats, counts {pc, pp, visits}). Returns 0 or -1. */
int oracle_bh_recursive(const uint64_t *sorted_keys, const float *ps, int64_t n, int32_t leaf_cap,
                        float side, float theta, float eps, float *acc, uint32_t *counts)
{
    if (n <= 0) return 0;
    pnode *root = pbuild(sorted_keys, ps, 0, n, 0, leaf_cap);
    if (!root) return -1;
    float theta2 = theta * theta, eps2 = eps * eps;
    for (int64_t i = 0; i < n; ++i) {
        float xi[3] = {ps[4 * i], ps[4 * i + 1], ps[4 * i + 2]};
        float a[3] = {0.0f, 0.0f, 0.0f};
        uint32_t cnt[3] = {0, 0, 0};
        pwalk(root, ps, i, xi, side, theta2, eps2, a, cnt);
        for (int c = 0; c < 3; ++c) {
            acc[3 * i + c] = a[c];
            counts[3 * i + c] = cnt[c];
        }
    }
    pfree(root);
    return 0;
}
