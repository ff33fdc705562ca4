/*
 * orrery_bh.h -- C ABI of the GB300 Barnes-Hut monopole force evaluation.
 *
 * One call evaluates softened gravitational accelerations for n particles with
 * a stackless depth-first octree and escape indices, as the orrery pages
 * describe it:
 *   - "sycl_tree_solver.hpp" reference page, Detailed Description: the walk,
 *     the gather into tree order and the scatter back to the caller's order,
 *     and the TreeTraversal enumeration {kIndependent, kCoherent};
 *   - "ADR-0029: Mask the accepted cells rather than descending together",
 *     Decision: the coherent walk advances each warp to the smallest node
 *     index any lane still wants, so every target is summed over exactly the
 *     nodes its own walk visits, in the same order;
 *   - "docs/performance/sycl_tree.md", "The machine and the device" table:
 *     softening, opening angle, leaf capacity, monopole only; "The divergence
 *     mitigation": what a node visit is.
 *
 * Arithmetic (both traversals, every step): IEEE binary32, round to nearest.
 *   cube:      lo_a = min x_a; side = max_a (max x_a - lo_a); inv = 2^21 / side
 *   key:       q_a = min(floor((x_a - lo_a) * inv), 2^21 - 1), bits of x, y, z
 *              interleaved x-high into a 63-bit Morton key
 *   sort:      stable on (key, original index)
 *   tree:      a cell is split iff it holds more than leaf_cap particles and
 *              its level is below 21; one child per non-empty octant, in
 *              octant order; nodes in depth-first preorder
 *   moments:   leaf M = sum m, S = sum fma(m, x, S) in sorted order; internal
 *              nodes sum their children in order; CoM = S / M (0 if M <= 0)
 *   criterion: accept iff (side 2^-L)^2 < (theta^2) * d2, d2 = |CoM - x_i|^2
 *              formed as fma(dz, dz, fma(dy, dy, dx * dx))
 *   term:      the workloads' softened law a_i += m (x_src - x_i) /
 *              (r^2 + eps^2)^(3/2), G = 1, over the target's own accepted
 *              cells (M, CoM) and opened leaves' particles j != i, in
 *              single precision. The kernels form r2 = d2 + eps^2 and
 *              y = 1/sqrt(r2) by a fixed recipe (the bit-level seed
 *              0x5f375a86 - bits(r2)/2 of C. Lomont, 2003, and three
 *              Newton-Raphson steps, within 2 ulp) or, with
 *              ORRERY_FAST_TERM, by the hardware approximation; then
 *              f = (m y)(y y) and a_i += f (x_src - x_i) by fused
 *              multiply-add. Each target's summation order depends only on
 *              the tree. Against the law evaluated plainly in binary32
 *              (m / (r2 sqrt(r2))) every target is within 1e-5 relative
 *              error on softened Plummer inputs (measured at most a few
 *              1e-6); where a target's terms nearly cancel the deviation is
 *              a few 1e-7 of the summed magnitude of its terms instead.
 * The acceptance tests, and so the interaction and visit counts, do not
 * depend on the term: they are exact, equal to a CPU restatement of the
 * steps above bit for bit. Every traversal except the descend-together
 * contrast gives the same counts; the independent and the coherent walks of
 * width 16, 32 and 64 also the same accelerations, bit for bit.
 *
 * Memory: every pointer named *_d or documented "device" is a CUDA device
 * pointer on the current device, owned by the caller. The library owns a
 * grow-only scratch workspace per device (released by orrery_bh_release).
 * Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 * stream); each call blocks once at its end to read back a status word, so
 * a call cannot be recorded into the caller's own stream capture (the
 * library captures and replays its own CUDA graphs). Calls on one device
 * are serialised by that device's lock; calls on different devices run
 * concurrently.
 *
 * Errors: a negative status; on any non-zero status the outputs are undefined.
 */
#ifndef ORRERY_BH_H
#define ORRERY_BH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORRERY_OK 0
#define ORRERY_EINVAL (-1)     /* bad argument; nothing was launched */
#define ORRERY_ENONFINITE (-2) /* a position or mass is NaN or infinite, a coordinate
                                  has magnitude 2^125 or more, or a cell's mass moments
                                  overflow binary32 (the supported range keeps every
                                  separation the walk forms finite) */
#define ORRERY_ERANGE (-3)     /* node count or size beyond the int32 range */
#define ORRERY_ECUDA (-4)      /* a CUDA runtime call failed */
#define ORRERY_EWALK (-5)      /* a walk exceeded its iteration bound */
#define ORRERY_ENOMEM (-6)     /* the workspace could not be allocated (the environment
                                  variable ORRERY_FAIL_ALLOC=1 forces this whenever the
                                  workspace has to grow, to test callers' failure paths) */
#define ORRERY_EINTERNAL (-7)  /* an index failed a device-side consistency check,
                                  or a bounded wait of the sort ran out; the access
                                  or the wait was skipped (a library defect; the
                                  environment variable ORRERY_TEST_SORT_STALL=1
                                  forces the wait to run out, for failure-path
                                  tests) */
#define ORRERY_ESCRATCH (-8)   /* orrery_bh_forces_noalloc: the problem does not fit
                                  its fixed scratch array */

/* Which traversal the walk kernel runs ("sycl_tree_solver.hpp", enum
 * TreeTraversal {kIndependent, kCoherent}; the coherent walk as ADR-0029,
 * Decision, defines it). Values 0-3 and 5 compute the same function of the input; the
 * coherent ones differ only in how many consecutive sorted targets share one
 * node index (the coherence width; docs/performance/sycl_tree.md, "The
 * sub-group width"), which changes the visit counts they report and their
 * speed. Value 4 is the published scheme the pages reject (ADR-0029,
 * Alternatives considered): a warp descends wherever any of its 32 targets
 * must, and accepts a cell only when all do, so a target's sum depends on
 * its warp-mates. It is kept to measure that contrast, not for use. */
typedef enum {
    ORRERY_INDEPENDENT = 0,       /* one thread per target, each on its own node index */
    ORRERY_COHERENT = 1,          /* 32 targets (one warp) share a node index */
    ORRERY_COHERENT_16 = 2,       /* 16 targets (half a warp) share a node index */
    ORRERY_COHERENT_64 = 3,       /* 64 targets (one warp, two per lane, packed float2
                                     arithmetic) share a node index: the fastest */
    ORRERY_DESCEND_TOGETHER = 4,  /* comparison only: group-dependent answer */
    ORRERY_COHERENT_BALLOT = 5    /* as ORRERY_COHERENT, next node by vote + escape
                                     instead of a minimum reduction (same visits) */
} orrery_traversal;

/* Flag ORed into the traversal argument: the force term's inverse square
 * root uses the hardware approximation (rsqrt.approx) instead of the fixed
 * Newton sequence. The width-64 walk is then ~20 % faster; acceptance
 * decisions, counts and visits are unchanged, and accelerations stay within
 * the same bounds against the plainly evaluated law (see the file head).
 * Without the flag the term is a fixed sequence of IEEE-754 binary32
 * operations, so the accelerations are reproducible bit for bit on any
 * IEEE-754 CPU that repeats them. */
#define ORRERY_FAST_TERM 0x100

/* Where the last evaluation spent its time ("sycl_tree_solver.hpp",
 * SyclTreeTimings), measured with CUDA events on the call's stream. */
typedef struct {
    float h2d_ms;     /* orrery_bh_forces_host only: host-to-device copies */
    float bbox_ms;    /* bounding cube reduction */
    float morton_ms;  /* quantise + interleave (above 4096 particles also the
                         digit counts of every radix pass) */
    float sort_ms;    /* radix sort of (key, index) */
    float gather_ms;  /* particles into tree order */
    float build_ms;   /* octree nodes and escape indices */
    float moments_ms; /* upward mass / centre-of-mass pass */
    float walk_ms;    /* the traversal, which also writes the results back to
                         the caller's order (the scatter is fused into it) */
    float scatter_ms; /* 0: fused into walk_ms */
    float d2h_ms;     /* orrery_bh_forces_host only: device-to-host copies */
    float total_ms;   /* first event to last */
    int32_t traversal;
    int32_t depth;       /* deepest node level */
    int64_t n;
    int64_t num_nodes;
    uint64_t launches;   /* kernels launched by that call */
} orrery_bh_timings;

/*
 * Evaluates accelerations for n particles: one force evaluation of the pages'
 * solver ("sycl_tree_solver.hpp", Detailed Description: the particles are
 * gathered into tree order, every target walks the octree, the results are
 * scattered back to the caller's order), with every phase on the device.
 *   pos_d        device, float32 [n][3] contiguous (x, y, z per particle)
 *   mass_d       device, float32 [n]
 *   n            0 <= n <= 2^30; n == 0 returns ORRERY_OK and launches nothing
 *   theta        opening angle, >= 0 (0 opens every cell: direct summation)
 *   eps          Plummer softening length, >= 0
 *   leaf_cap     >= 1: a cell holding at most this many particles is a leaf
 *   traversal    an orrery_traversal value, optionally | ORRERY_FAST_TERM
 *   acc_d        device, float32 [n][3], written in the caller's order
 *   interactions_d  device, uint32 [n][2] {particle-cell, particle-particle}
 *                per target in the caller's order, or NULL
 *   visits_d     device, uint32 [n] node visits per target, or NULL. For the
 *                independent walk a target's own walk; for a coherent walk
 *                the size of the union of its group's walks (the group =
 *                16, 32 or 64 consecutive sorted targets)
 *   stream       cudaStream_t
 * Returns ORRERY_OK or a negative status.
 */
int orrery_bh_forces(const float *pos_d, const float *mass_d, int64_t n, float theta, float eps,
                     int32_t leaf_cap, int32_t traversal, float *acc_d, uint32_t *interactions_d,
                     uint32_t *visits_d, void *stream);

/*
 * orrery_bh_forces for a slice of the targets: the tree is built over all n
 * particles (every particle is a source), and only the targets at SORTED
 * positions [begin, end) are walked. Targets are independent once the tree
 * exists ("sycl_tree_solver.hpp", "What is not given up": each target is
 * summed over its own walk), so disjoint slices that cover [0, n) give,
 * together, exactly the full evaluation: the unit a caller shards across
 * devices or streams. Sorted positions are the Morton order of the particles
 * (the permutation orrery_bh_tree returns); callers need not know it, only
 * that equal slices of [0, n) partition the targets.
 *   begin, end   0 <= begin <= end <= n, else ORRERY_EINVAL; begin == end
 *                builds the tree and walks nothing
 *   acc_d, interactions_d, visits_d  as in orrery_bh_forces, but only the
 *                slice's targets are written (at their caller-order
 *                positions); every other entry is left as it was
 * Accelerations and interaction counts equal those of the full evaluation
 * for every slice. Visit counts of a coherent traversal equal them when
 * begin and end are multiples of the group width (end may also be n);
 * otherwise the groups are formed from begin onward, so each count is the
 * union over other neighbours (never below the target's own walk). The
 * descend-together traversal's sums depend on the groups too.
 */
int orrery_bh_forces_range(const float *pos_d, const float *mass_d, int64_t n, float theta,
                           float eps, int32_t leaf_cap, int32_t traversal, int64_t begin,
                           int64_t end, float *acc_d, uint32_t *interactions_d, uint32_t *visits_d,
                           void *stream);

/*
 * The same evaluation from and to HOST memory (page-locked memory gives the
 * fastest copies; pageable memory works). The input copies run on `stream`
 * inside the call; pos, mass and acc are required, interactions and visits
 * may be NULL. Shapes and order as in orrery_bh_forces. An output buffer that
 * is page-locked over its whole extent (cudaHostAlloc, cudaHostRegister) is
 * written by the walk directly, over the host link while the walk runs; a
 * pageable one is filled by a copy after the walk. Either way its contents
 * are final when the call returns (the call blocks), and d2h_ms in the
 * timings covers only the copies made.
 */
int orrery_bh_forces_host(const float *pos, const float *mass, int64_t n, float theta, float eps,
                          int32_t leaf_cap, int32_t traversal, float *acc, uint32_t *interactions,
                          uint32_t *visits, void *stream);

/*
 * The same evaluation as orrery_bh_forces, for callers that must not allocate
 * device memory during a call: host applications or plugins that own every
 * device allocation themselves, code that runs while a CUDA graph may be
 * under capture, and latency-critical loops that cannot take the implicit
 * device synchronisation of cudaMalloc / cudaFree. (The pages have no
 * counterpart: their solver allocates its shared-memory buffers per call.)
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine. Its scratch
 * is one fixed 16 MiB array inside the library's device code, which every GPU
 * that loads the library holds until the process exits. A call fits iff its
 * buffers fit 16 MiB: at leaf_cap >= 16 every n <= 65536 fits; at leaf_cap 32
 * every n <= 80000 fits. A call that does not fit returns ORRERY_ESCRATCH
 * before launching anything.
 *
 * Every call looks up the array's device address on the caller's current
 * device (so a context torn down by cudaDeviceReset and created again is
 * handled). The first call on a device may load the library's device code
 * there and sets kernel attributes: make it before any stream capture. All
 * calls share the array, which keeps the previous call's contents; each call
 * clears what must start at zero. Calls whose GPU work overlapped would race
 * on the array: this entry point serialises its calls and waits for its own
 * work before returning, so its calls do not overlap.
 *
 * Each call ends by copying a status word to the host and synchronising
 * `stream`. If another thread may be capturing a CUDA graph meanwhile, pass a
 * stream created with cudaStreamNonBlocking (not the legacy NULL stream),
 * and have the capturing thread use cudaStreamCaptureModeThreadLocal or
 * cudaStreamCaptureModeRelaxed: under the global mode a synchronising call
 * from another thread invalidates that capture.
 * Arguments, layouts, results and statuses as in orrery_bh_forces; no phase
 * timings are recorded.
 */
int orrery_bh_forces_noalloc(const float *pos_d, const float *mass_d, int64_t n, float theta,
                             float eps, int32_t leaf_cap, int32_t traversal, float *acc_d,
                             uint32_t *interactions_d, uint32_t *visits_d, void *stream);

/*
 * Runs the cube, key, sort, gather, build and moments steps and copies their
 * results out (for inspection and tests). Every output is a device pointer
 * and may be NULL:
 *   cube_d       float32 [5] {lo_x, lo_y, lo_z, side, inv}
 *   keys_d       uint64 [n] Morton keys in sorted order
 *   perm_d       uint32 [n] original index of each sorted slot
 *   nodes_d      int32 [max_nodes][4] {escape, first, count, level}, preorder
 *   com_d        float32 [max_nodes][4] {CoM_x, CoM_y, CoM_z, M}
 *   num_nodes    host int64, the node count (required)
 * Returns ORRERY_ERANGE when max_nodes is below the node count (num_nodes is
 * still set).
 */
int orrery_bh_tree(const float *pos_d, const float *mass_d, int64_t n, int32_t leaf_cap,
                   float *cube_d, uint64_t *keys_d, uint32_t *perm_d, int32_t *nodes_d,
                   float *com_d, int64_t max_nodes, int64_t *num_nodes, void *stream);

/*
 * Direct summation over every pair, the solver the pages time the tree
 * against (docs/performance/sycl_tree.md, "Against the two solvers it has to
 * beat"): acc_i = sum over j != i, j ascending in caller order, of the tree's
 * particle term (same softening and arithmetic, no approximation). O(n^2).
 *   pos_d [n][3], mass_d [n], acc_d [n][3]: device float32, caller order.
 * Returns ORRERY_OK, ORRERY_EINVAL, ORRERY_ENONFINITE (here only for a NaN or
 * infinite position or mass: the range limit of the tree does not apply) or
 * ORRERY_ECUDA.
 */
int orrery_direct_forces(const float *pos_d, const float *mass_d, int64_t n, float eps,
                         float *acc_d, void *stream);

/* Upper bound of the node count for n particles and a leaf capacity:
 * n + 21 * floor(n / (leaf_cap + 1)) + 1 (leaves are disjoint and non-empty;
 * internal cells of one level are disjoint and hold more than leaf_cap).
 * Returns -1 for invalid arguments. */
int64_t orrery_bh_max_nodes(int64_t n, int32_t leaf_cap);

/* The FP32 fused multiply-add rate this GPU delivers, measured: long
 * independent FMA chains on every SM, scalar (FFMA) and packed (FFMA2, two
 * FMAs per lane per instruction, the form the walk's arithmetic uses), each
 * timed with CUDA events over one launch after an untimed one (about 15 ms
 * each on a GB300). The walk is bound by plain FP32 arithmetic, so this is
 * its measured roofline denominator beside the nominal SMs x 128 lanes x 2
 * flops x clock. Work is enqueued on `stream` (a cudaStream_t, NULL for the
 * default stream) and the call blocks until it is done; calls are serialised.
 *   tflops_scalar, tflops_packed: host outputs, TFLOP/s (an FMA = 2 flops).
 *   sm_mhz: host output or NULL: the SM clock during the scalar probe (each
 *           block's clock cycles over the launch's elapsed time, median).
 * Returns ORRERY_OK, ORRERY_EINVAL (a null rate output) or ORRERY_ECUDA. */
int orrery_fp32_fma_rate(double *tflops_scalar, double *tflops_packed, double *sm_mhz,
                         void *stream);

/* Copies the phase timings of the last successful evaluation on this process. */
int orrery_bh_last_timings(orrery_bh_timings *out);

/* Total kernels this library has launched in this process. */
uint64_t orrery_bh_kernel_launches(void);

/* A static string describing a status code. */
const char *orrery_bh_strerror(int status);

/* Frees the workspaces of every device this process used. */
void orrery_bh_release(void);

#ifdef __cplusplus
}
#endif

#endif /* ORRERY_BH_H */
