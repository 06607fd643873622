// ra_api.cu - the C ABI of libra: argument checks, the ring schedule, kernel dispatch,
// the device error word.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "ra_internal.cuh"

namespace ra {
cudaError_t launch_attn_simt(const StepParams &P, int blocks_y, cudaStream_t stream);
cudaError_t launch_attn_tc(const StepParams &P, int blocks_y, int num_sms, cudaStream_t stream);
int attn_tc_rows_per_block();
cudaError_t launch_wait_selftest(int64_t limit_ns, int *err, cudaStream_t stream);
cudaError_t launch_bounds_selftest(int *err, cudaStream_t stream);

cudaError_t launch_lse_merge(const MergeParams &P, int num_sms, cudaStream_t stream);
cudaError_t launch_attn_bwd_simt(const BwdParams &P, int parts, cudaStream_t stream);
cudaError_t launch_bwd_rowdot(const BwdParams &P, int num_sms, cudaStream_t stream);
cudaError_t launch_ulysses(const UlyssesParams &P, int num_sms, cudaStream_t stream);
cudaError_t launch_attn_bwd_tc(const BwdParams &P, int parts, int num_sms, int64_t wait_ns, int *err,
                               cudaStream_t stream, bool after_dq);
cudaError_t launch_fill_identity(void *o, int o_bf16, const int64_t *so, float *lse, int B, int H,
                                 int N, int D, int r0, int r1, int num_sms, cudaStream_t stream);
}  // namespace ra

using namespace ra;

// ---------------------------------------------------------------- error state

static thread_local std::string t_last_error;
static thread_local int64_t t_launches = 0;

static ra_status fail(ra_status s, const std::string &msg) {
    t_last_error = msg;
    return s;
}

// Launch failures injected on the host (ra_debug_fail_next_launches): the next n kernel
// launches of the calling thread report cudaErrorLaunchFailure without reaching the GPU.
static thread_local int t_inject_launch_failures = 0;
static thread_local bool t_injected = false;

// Guard in front of every kernel launch: true when this launch is to fail (injected).
static bool launch_injected() {
    if (t_inject_launch_failures <= 0) return false;
    --t_inject_launch_failures;
    t_injected = true;
    return true;
}

// Per-launch timing (ra_debug_time_launches): while on, each kernel launch of the calling
// thread is bracketed by two CUDA events on its stream.
struct TimedLaunch {
    const char *name;
    cudaEvent_t start, stop;
};
static thread_local bool t_time_launches = false;
static thread_local std::vector<TimedLaunch> t_timed;

// Every kernel launch goes through here: an injected failure, or the launch `f` (timed
// when timing is on).
template <class F>
static cudaError_t guarded_launch(const char *name, cudaStream_t st, F &&f) {
    if (launch_injected()) return cudaErrorLaunchFailure;
    if (!t_time_launches) return f();
    TimedLaunch t{name, nullptr, nullptr};
    if (cudaEventCreate(&t.start) != cudaSuccess || cudaEventCreate(&t.stop) != cudaSuccess ||
        cudaEventRecord(t.start, st) != cudaSuccess) {
        if (t.start) cudaEventDestroy(t.start);
        if (t.stop) cudaEventDestroy(t.stop);
        return f();
    }
    const cudaError_t e = f();
    if (cudaEventRecord(t.stop, st) == cudaSuccess) {
        t_timed.push_back(t);
    } else {
        cudaEventDestroy(t.start);
        cudaEventDestroy(t.stop);
    }
    return e;
}

static ra_status cuda_fail(cudaError_t e, const char *what) {
    std::string msg = std::string(what) + ": " + cudaGetErrorString(e);
    if (t_injected) msg += " (injected on the host by ra_debug_fail_next_launches)";
    t_injected = false;
    return fail(RA_ERR_CUDA, msg);
}

__device__ int g_device_error;

// Work counter pairs of the tensor-core forward launches (next item, CTAs finished), used in
// rotation: a launch takes the next pair, and its last CTA zeroes the pair again; a pair is
// reused only kSchedSlots launches later, after that launch has long finished.
constexpr int kSchedSlots = 1024;
__device__ int g_sched[2 * kSchedSlots];

static const int kMaxDev = 64;
static const int kHostGroups = 8;  // head groups of the host-buffer pipeline (at most)
static std::mutex g_mu;
static int *g_err_ptr[kMaxDev];
static int *g_sched_ptr[kMaxDev];
static uint32_t g_sched_seq[kMaxDev];
static int g_num_sms[kMaxDev];
static int64_t g_wait_limit_ns = 2000000000LL;
static int64_t g_producer_delay_ns = 0;

struct DevInfo {
    int dev;
    int *err;
    int sms;
    bool tc_ok;
};

// The work counter pair of the next tensor-core forward launch on `dev`.
static int *next_sched(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sched_ptr[dev]) return nullptr;
    return g_sched_ptr[dev] + 2 * (g_sched_seq[dev]++ % kSchedSlots);
}

static bool device_info(DevInfo &d, std::string &msg) {
    if (cudaGetDevice(&d.dev) != cudaSuccess || d.dev < 0 || d.dev >= kMaxDev) {
        msg = "no current CUDA device";
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[d.dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_device_error);
        if (e != cudaSuccess) {
            msg = std::string("cudaGetSymbolAddress(error word): ") + cudaGetErrorString(e);
            return false;
        }
        void *ps = nullptr;
        e = cudaGetSymbolAddress(&ps, g_sched);
        if (e != cudaSuccess) {
            msg = std::string("cudaGetSymbolAddress(work counters): ") + cudaGetErrorString(e);
            return false;
        }
        g_sched_ptr[d.dev] = static_cast<int *>(ps);
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d.dev);
        g_num_sms[d.dev] = sms > 0 ? sms : 1;
        g_err_ptr[d.dev] = static_cast<int *>(p);
    }
    d.err = g_err_ptr[d.dev];
    d.sms = g_num_sms[d.dev];
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d.dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d.dev);
    d.tc_ok = (major == 10 && minor == 3);
    return true;
}

// ---------------------------------------------------------------- argument checks

static bool is_dtype(int32_t d) { return d == RA_F32 || d == RA_BF16; }
static int esize(int32_t d) { return d == RA_F32 ? 4 : 2; }

static ra_status check_tensor(const ra_tensor *t, const char *name) {
    if (!t) return fail(RA_ERR_INVALID_ARG, std::string(name) + " is NULL");
    if (!is_dtype(t->dtype)) return fail(RA_ERR_INVALID_ARG, std::string(name) + ": bad dtype");
    for (int i = 0; i < 4; ++i)
        if (t->shape[i] < 0) return fail(RA_ERR_INVALID_ARG, std::string(name) + ": negative shape");
    const int64_t numel = t->shape[0] * t->shape[1] * t->shape[2] * t->shape[3];
    if (numel > 0) {
        if (!t->data) return fail(RA_ERR_INVALID_ARG, std::string(name) + ": data is NULL");
        if (t->stride[3] != 1)
            return fail(RA_ERR_INVALID_ARG, std::string(name) + ": stride[3] must be 1");
        for (int i = 0; i < 3; ++i)
            if (t->stride[i] < 0)
                return fail(RA_ERR_INVALID_ARG, std::string(name) + ": negative stride");
        if (reinterpret_cast<uintptr_t>(t->data) % esize(t->dtype))
            return fail(RA_ERR_INVALID_ARG, std::string(name) + ": misaligned data pointer");
    }
    return RA_OK;
}

static bool aligned16(const ra_tensor *t) {
    const int64_t per16 = 16 / esize(t->dtype);
    return reinterpret_cast<uintptr_t>(t->data) % 16 == 0 && t->stride[0] % per16 == 0 &&
           t->stride[1] % per16 == 0 && t->stride[2] % per16 == 0;
}

struct Problem {
    int64_t B, Hq, Hkv, N, D;
    int32_t dtype;
};

static ra_status check_qkvo(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                            const ra_tensor *o, const float *lse, Problem &pb, bool need_lse = true) {
    ra_status s;
    if ((s = check_tensor(q, "q")) || (s = check_tensor(k, "k")) || (s = check_tensor(v, "v")) ||
        (s = check_tensor(o, "o")))
        return s;
    pb.B = q->shape[0];
    pb.Hq = q->shape[1];
    pb.N = q->shape[2];
    pb.D = q->shape[3];
    pb.Hkv = k->shape[1];
    pb.dtype = q->dtype;
    if (k->dtype != q->dtype || v->dtype != q->dtype || o->dtype != q->dtype)
        return fail(RA_ERR_INVALID_ARG, "q, k, v, o must share one dtype");
    for (int i = 0; i < 4; ++i) {
        if (k->shape[i] != v->shape[i]) return fail(RA_ERR_INVALID_ARG, "k and v shapes differ");
        if (o->shape[i] != q->shape[i]) return fail(RA_ERR_INVALID_ARG, "o shape differs from q");
    }
    if (k->shape[0] != pb.B || k->shape[2] != pb.N || k->shape[3] != pb.D)
        return fail(RA_ERR_INVALID_ARG, "k/v must be [B, Hkv, N, D] with q's B, N, D");
    const int64_t rows = pb.B * pb.Hq * pb.N;
    if (rows == 0) return RA_OK;
    if (pb.Hkv < 1 || pb.Hq % pb.Hkv != 0)
        return fail(RA_ERR_INVALID_ARG, "Hq must be a positive multiple of Hkv");
    if (pb.D < 1) return fail(RA_ERR_INVALID_ARG, "D must be >= 1");
    if (need_lse && !lse) return fail(RA_ERR_INVALID_ARG, "lse is NULL");
    if (pb.D > 128) return fail(RA_ERR_UNSUPPORTED, "head size D > 128 is not supported");
    if (pb.N > (int64_t)1 << 30 || pb.B * pb.Hq > 65535LL * 32768LL)
        return fail(RA_ERR_UNSUPPORTED, "problem too large for one launch grid");
    return RA_OK;
}

// ---------------------------------------------------------------- ring schedule

struct Range {
    int64_t a, b;
};

// Row ranges of rank r under the contiguous or zigzag layout, into out[0..2); returns how
// many (1 or 2).  No allocation: the allocation-free entry point plans with it too.
static int rank_ranges(int64_t N, int R, int layout, int r, Range out[2]) {
    if (layout == RA_LAYOUT_CONTIG) {
        const int64_t c = N / R;
        out[0] = {r * c, (r + 1) * c};
        return 1;
    }
    const int64_t h = N / (2 * (int64_t)R);
    out[0] = {r * h, (r + 1) * h};
    out[1] = {(2 * (int64_t)R - 1 - r) * h, (2 * (int64_t)R - r) * h};
    return 2;
}

// Whether rank r's query chunk ending at row q1 - 1 sees any key of the block it holds at
// `step` (that of rank (r - step) mod R).  Striped layout: every rank's rows are [0, N/R)
// of its interleave, and under causality a later rank's block is seen from row index 1.
static bool chunk_touched(int64_t N, int R, int layout, int causal, int step, int r, int64_t q1) {
    const int j = ((r - step) % R + R) % R;
    if (layout == RA_LAYOUT_STRIPED) {
        const int64_t c = N / R;
        return c > 0 && !(causal && j > r && c < 2);
    }
    Range kv[2];
    const int nk = rank_ranges(N, R, layout, j, kv);
    for (int i = 0; i < nk; ++i) {
        if (kv[i].b <= kv[i].a) continue;
        if (causal && kv[i].a > q1 - 1) continue;  // every key after every row
        return true;
    }
    return false;
}

static int64_t seg_keys(const Seg &x) { return (int64_t)(x.k1[0] - x.k0[0]) + (x.k1[1] - x.k0[1]); }

// The segments of one ring step into segs[0 .. 2R): for every rank r, each of its query
// chunks against the chunks of rank (r - step) mod R that some row of the chunk can see,
// flagged SEG_FIRST when no earlier step touches the chunk and SEG_FINAL when no later one
// does, heaviest (most keys) first, equal ones in rank order.  Striped layout: rank r holds
// positions r, r + R, r + 2R, ...; its segment is indices [0, N/R) of the interleave
// against the same indices of rank j, with key index j' visible to row index i iff
// j' + [j > r] <= i under causality.  Returns the number of segments.  No allocation
// (a stable insertion sort), so the allocation-free entry point shares this schedule.
static int plan_step(int64_t N, int R, int layout, int causal, int step, Seg *segs) {
    int n = 0;
    for (int r = 0; r < R; ++r) {
        const int j = ((r - step) % R + R) % R;
        Seg cand[2];
        int nc = 0;
        if (layout == RA_LAYOUT_STRIPED) {
            const int64_t c = N / R;
            Seg &g = cand[0];
            memset(&g, 0, sizeof g);
            g.q0 = 0;
            g.q1 = (int32_t)c;
            g.k0[0] = 0;
            g.k1[0] = (int32_t)c;
            g.k0[1] = g.k1[1] = (int32_t)c;
            g.rank = r;
            g.q_rank = r;
            g.kv_rank = j;
            g.diag = (causal && j > r) ? 1 : 0;
            if (!(c == 0 || (causal && g.diag > c - 1))) nc = 1;  // else no row sees a key
        } else {
            Range qr[2], kv[2];
            const int nq = rank_ranges(N, R, layout, r, qr);
            const int nkv = rank_ranges(N, R, layout, j, kv);
            for (int qi = 0; qi < nq; ++qi) {
                if (qr[qi].b <= qr[qi].a) continue;
                Seg &g = cand[nc];
                memset(&g, 0, sizeof g);
                g.q0 = (int32_t)qr[qi].a;
                g.q1 = (int32_t)qr[qi].b;
                int nk = 0;
                for (int ki = 0; ki < nkv; ++ki) {
                    if (kv[ki].b <= kv[ki].a) continue;
                    if (causal && kv[ki].a > qr[qi].b - 1) continue;  // every key after every row
                    g.k0[nk] = (int32_t)kv[ki].a;
                    g.k1[nk] = (int32_t)kv[ki].b;
                    ++nk;
                }
                if (nk == 0) continue;
                if (nk == 1) g.k0[1] = g.k1[1] = g.k1[0];
                g.rank = r;
                ++nc;
            }
        }
        for (int i = 0; i < nc; ++i) {
            Seg g = cand[i];
            bool earlier = false, later = false;
            for (int t = 0; t < step && !earlier; ++t) earlier = chunk_touched(N, R, layout, causal, t, r, g.q1);
            for (int t = step + 1; t < R && !later; ++t) later = chunk_touched(N, R, layout, causal, t, r, g.q1);
            g.flags = (earlier ? 0 : SEG_FIRST) | (later ? 0 : SEG_FINAL);
            // heaviest segments first (more keys), so they lead every dispatch round
            int at = n;
            while (at > 0 && seg_keys(segs[at - 1]) < seg_keys(g)) {
                segs[at] = segs[at - 1];
                --at;
            }
            segs[at] = g;
            ++n;
        }
    }
    return n;
}

static ra_status check_ring(int64_t N, int R, int layout) {
    if (R < 1) return fail(RA_ERR_INVALID_ARG, "ring_size must be >= 1");
    if (layout != RA_LAYOUT_CONTIG && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIPED)
        return fail(RA_ERR_INVALID_ARG, "unknown layout");
    if ((layout == RA_LAYOUT_CONTIG || layout == RA_LAYOUT_STRIPED) && N % R != 0)
        return fail(RA_ERR_INVALID_ARG, "contiguous and striped layouts need N % ring_size == 0");
    if (layout == RA_LAYOUT_ZIGZAG && N % (2 * (int64_t)R) != 0)
        return fail(RA_ERR_INVALID_ARG, "zigzag layout needs N % (2 ring_size) == 0");
    return RA_OK;
}

// ---------------------------------------------------------------- ring backward schedule

// One block of a backward ring step: rank r's query chunk qr against chunk kr of the rank
// j = (r - step) mod R whose keys and values r holds at that step.
struct BPair {
    int r, j;
    Range qr, kr;
    int diag;
};

// The blocks of one step with at least one visible (row, key) pair: the same visibility
// as the forward's step (causal on global positions; the striped interleave's offset).
static void bwd_pairs(int64_t N, int R, int layout, int causal, int step, std::vector<BPair> &out) {
    out.clear();
    for (int r = 0; r < R; ++r) {
        const int j = ((r - step) % R + R) % R;
        if (layout == RA_LAYOUT_STRIPED) {
            const int64_t c = N / R;
            const int diag = (causal && j > r) ? 1 : 0;
            if (c == 0 || (causal && diag > c - 1)) continue;
            out.push_back({r, j, {0, c}, {0, c}, diag});
            continue;
        }
        Range qrs[2], krs[2];
        const int nq = rank_ranges(N, R, layout, r, qrs), nk = rank_ranges(N, R, layout, j, krs);
        for (int qi = 0; qi < nq; ++qi)
            for (int ki = 0; ki < nk; ++ki) {
                const Range &qr = qrs[qi], &kr = krs[ki];
                if (qr.b <= qr.a || kr.b <= kr.a) continue;
                if (causal && kr.a > qr.b - 1) continue;  // every key after every row
                out.push_back({r, j, qr, kr, 0});
            }
    }
}

// A step's blocks grouped by fixed range: by query chunk for the dQ kernels (the chunk
// stays on its rank), by key chunk for the dK/dV kernels (the chunk's gradients go back
// to its rank).  `owner` receives the rank that owns each segment's fixed range.
static void bwd_group(const std::vector<BPair> &pairs, bool dq, bool striped, std::vector<BSeg> &segs,
                      std::vector<int> &owner) {
    segs.clear();
    owner.clear();
    for (const BPair &p : pairs) {
        const int frank = dq ? p.r : p.j, srank = dq ? p.j : p.r;
        const Range &f = dq ? p.qr : p.kr;
        const Range &sr = dq ? p.kr : p.qr;
        size_t i = 0;
        while (i < segs.size() && !(owner[i] == frank && segs[i].f0 == f.a)) ++i;
        if (i == segs.size()) {
            BSeg g;
            memset(&g, 0, sizeof g);
            g.f0 = (int32_t)f.a;
            g.f1 = (int32_t)f.b;
            g.s0[0] = (int32_t)sr.a;
            g.s1[0] = (int32_t)sr.b;
            g.s0[1] = g.s1[1] = (int32_t)sr.b;
            g.f_rank = striped ? frank : 0;
            g.s_rank = striped ? srank : 0;
            g.diag = p.diag;
            segs.push_back(g);
            owner.push_back(frank);
        } else {  // a second chunk of the partner rank (zigzag): ranges kept in order
            BSeg &g = segs[i];
            if (sr.a < g.s0[0]) {
                g.s0[1] = g.s0[0];
                g.s1[1] = g.s1[0];
                g.s0[0] = (int32_t)sr.a;
                g.s1[0] = (int32_t)sr.b;
            } else {
                g.s0[1] = (int32_t)sr.a;
                g.s1[1] = (int32_t)sr.b;
            }
        }
    }
}

static int64_t bseg_work(const BSeg &g) {
    return (int64_t)(g.s1[0] - g.s0[0]) + (g.s1[1] - g.s0[1]);
}

// The first and last step that writes each fixed range, per kind (0: dQ, 1: dK/dV),
// indexed by owner rank * 2 + chunk slot; then one step's segments with their flags,
// heaviest first.
struct BwdPlan {
    int64_t N;
    int R, layout, causal;
    std::vector<int> first[2], last[2];

    int slot(int own, int32_t f0) const {
        if (layout != RA_LAYOUT_ZIGZAG) return own * 2;
        return own * 2 + ((int64_t)f0 < (int64_t)(own + 1) * (N / (2 * (int64_t)R)) ? 0 : 1);
    }

    BwdPlan(int64_t n, int r, int lay, int c) : N(n), R(r), layout(lay), causal(c) {
        std::vector<BPair> pairs;
        std::vector<BSeg> segs;
        std::vector<int> owner;
        for (int kind = 0; kind < 2; ++kind) {
            first[kind].assign(2 * (size_t)R, -1);
            last[kind].assign(2 * (size_t)R, -1);
        }
        for (int step = 0; step < R; ++step) {
            bwd_pairs(N, R, layout, causal, step, pairs);
            for (int kind = 0; kind < 2; ++kind) {
                bwd_group(pairs, kind == 0, layout == RA_LAYOUT_STRIPED, segs, owner);
                for (size_t i = 0; i < segs.size(); ++i) {
                    const int sl = slot(owner[i], segs[i].f0);
                    if (first[kind][sl] < 0) first[kind][sl] = step;
                    last[kind][sl] = step;
                }
            }
        }
    }

    void step(int st, int kind, std::vector<BSeg> &segs) const {
        std::vector<BPair> pairs;
        std::vector<int> owner;
        bwd_pairs(N, R, layout, causal, st, pairs);
        bwd_group(pairs, kind == 0, layout == RA_LAYOUT_STRIPED, segs, owner);
        for (size_t i = 0; i < segs.size(); ++i) {
            const int sl = slot(owner[i], segs[i].f0);
            segs[i].flags = (first[kind][sl] == st ? SEG_FIRST : 0) | (last[kind][sl] == st ? SEG_FINAL : 0);
        }
        std::stable_sort(segs.begin(), segs.end(),
                         [](const BSeg &x, const BSeg &y) { return bseg_work(x) > bseg_work(y); });
    }
};

// The fused ring launch (tensor cores): one segment per query chunk, tagged with its
// rank; the kernel walks the chunk's key ranges of steps 0..R-1 in ring order (those of
// rank (r - s) mod R) and keeps the running result on chip, so each row is written once
// (SEG_FIRST | SEG_FINAL) and no float32 running output is needed.  Heaviest chunks (most
// visible keys over all steps) first.  Fills out[0 .. kMaxSeg) and returns the segment
// count, or 0 when the fused launch does not apply (more chunks than a launch holds; a
// striped rank that is not whole 128-row tiles).  No allocation.
static int fused_ring_segments(int64_t N, int R, int layout, int causal, Seg *out) {
    if (layout == RA_LAYOUT_STRIPED) {
        // one segment per rank, in the rank-local index space: the kernel walks each
        // step's causal prefix with its diagonal offset.  Needs whole 128-row tiles per
        // rank (every step of an item then has the same tile count); the ranks' work is
        // the same, so their order does not matter.
        const int64_t c = N / R;
        if (R > kMaxSeg || c % 128 != 0 || c > INT32_MAX || c == 0) return 0;
        for (int r = 0; r < R; ++r) {
            Seg &g = out[r];
            memset(&g, 0, sizeof g);
            g.q0 = 0;
            g.q1 = (int32_t)c;
            g.q_rank = r;
            g.rank = r;
            g.flags = SEG_FIRST | SEG_FINAL;
        }
        (void)causal;
        return R;
    }
    const int chunks = layout == RA_LAYOUT_ZIGZAG ? 2 * R : R;
    if (chunks > kMaxSeg || N > INT32_MAX) return 0;
    int64_t work[kMaxSeg];
    int n = 0;
    for (int r = 0; r < R; ++r) {
        Range qrs[2];
        const int nq = rank_ranges(N, R, layout, r, qrs);
        for (int qi = 0; qi < nq; ++qi) {
            const Range &qr = qrs[qi];
            if (qr.b <= qr.a) continue;
            Seg g;
            memset(&g, 0, sizeof g);
            g.q0 = (int32_t)qr.a;
            g.q1 = (int32_t)qr.b;
            g.rank = r;
            g.flags = SEG_FIRST | SEG_FINAL;
            int64_t keys = 0;
            for (int st = 0; st < R; ++st) {
                const int j = ((r - st) % R + R) % R;
                Range krs[2];
                const int nk = rank_ranges(N, R, layout, j, krs);
                for (int ki = 0; ki < nk; ++ki) {
                    const Range &kr = krs[ki];
                    if (kr.b <= kr.a || (causal && kr.a > qr.b - 1)) continue;
                    keys += kr.b - kr.a;
                }
            }
            int at = n;  // stable insertion, most keys first
            while (at > 0 && work[at - 1] < keys) {
                work[at] = work[at - 1];
                out[at] = out[at - 1];
                --at;
            }
            work[at] = keys;
            out[at] = g;
            ++n;
        }
    }
    return n;
}

// The fused ring backward (tensor cores, contiguous or zigzag layout): kind 0, one dQ
// segment per query chunk; kind 1, one dK/dV segment per key chunk; each tagged with its
// rank, the kernels walk the partner ranges of steps 0..R-1 and keep the gradient on
// chip, so each row is written once.  Heaviest first.  False when it does not apply.
static bool fused_bwd_segments(int64_t N, int R, int layout, int causal, int kind, std::vector<BSeg> &out) {
    out.clear();
    if (layout == RA_LAYOUT_STRIPED) {
        // one segment per rank in the rank-local index space; every step's partner tiles
        // follow from the rank and the step (the kernels' striped walk).  Needs whole
        // 128-row tiles per rank; the ranks' work is the same, so their order does not matter.
        const int64_t c = N / R;
        if (R > kMaxBSeg || c % 128 != 0 || c > INT32_MAX || c == 0) return false;
        for (int r = 0; r < R; ++r) {
            BSeg g;
            memset(&g, 0, sizeof g);
            g.f0 = 0;
            g.f1 = (int32_t)c;
            g.f_rank = g.s_rank = r;  // step 0: the rank's own keys and queries
            g.flags = SEG_FIRST | SEG_FINAL;
            g.rank = r;
            out.push_back(g);
        }
        (void)causal;
        (void)kind;
        return true;
    }
    const int chunks = layout == RA_LAYOUT_ZIGZAG ? 2 * R : R;
    if (chunks > kMaxBSeg || N > INT32_MAX) return false;
    std::vector<std::pair<int64_t, BSeg>> work;
    for (int r = 0; r < R; ++r) {
        Range frs[2];
        const int nf = rank_ranges(N, R, layout, r, frs);
        for (int fi = 0; fi < nf; ++fi) {
            const Range &f = frs[fi];
            if (f.b <= f.a) continue;
            BSeg g;
            memset(&g, 0, sizeof g);
            g.f0 = (int32_t)f.a;
            g.f1 = (int32_t)f.b;
            g.flags = SEG_FIRST | SEG_FINAL;
            g.rank = r;
            int64_t pairs = 0;
            for (int s = 0; s < R; ++s) {
                const int j = kind ? (r + s) % R : ((r - s) % R + R) % R;
                Range prs[2];
                const int np = rank_ranges(N, R, layout, j, prs);
                for (int pi = 0; pi < np; ++pi) {
                    const Range &p = prs[pi];
                    if (p.b <= p.a) continue;
                    if (causal && (kind ? f.a > p.b - 1 : p.a > f.b - 1)) continue;
                    pairs += p.b - p.a;
                }
            }
            work.push_back({pairs, g});
        }
    }
    std::stable_sort(work.begin(), work.end(),
                     [](const std::pair<int64_t, BSeg> &x, const std::pair<int64_t, BSeg> &y) { return x.first > y.first; });
    for (const auto &w : work) out.push_back(w.second);
    return !out.empty();
}

// ---------------------------------------------------------------- dispatch

// Query heads per group of consecutive single-block work items: a group's K and V (4 N D
// bytes per KV head in bf16) within kGroupKvBytes, so that they stay in the 129 MB L2 while
// the group's items run on the persistent grid; whole KV heads (G query heads) at least.
// 0 (no grouping) when every head fits at once.
constexpr double kGroupKvBytes = 48.0 * (1 << 20);
static int32_t head_group(const Problem &pb) {
    const int64_t G = pb.Hkv > 0 ? pb.Hq / pb.Hkv : 1;
    const double per_kv = 4.0 * (double)pb.N * (double)pb.D;
    const int64_t units = pb.B * pb.Hkv;  // (batch, KV head) units
    int64_t kv = (int64_t)(kGroupKvBytes / std::max(per_kv, 1.0));
    kv = std::max<int64_t>(kv, 1);
    if (kv >= units) return 0;
    return (int32_t)std::min<int64_t>(kv * G, 1 << 30);
}

static void fill_common(StepParams &P, const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                        const ra_tensor *o, float *lse, const Problem &pb, int causal,
                        float scale, const DevInfo &di) {
    memset(&P, 0, sizeof P);
    P.q = q->data;
    P.k = k->data;
    P.v = v->data;
    P.o = o->data;
    for (int i = 0; i < 3; ++i) {
        P.sq[i] = q->stride[i];
        P.sk[i] = k->stride[i];
        P.sv[i] = v->stride[i];
        P.so[i] = o->stride[i];
    }
    P.lse = lse;
    P.B = (int32_t)pb.B;
    P.Hq = (int32_t)pb.Hq;
    P.Hkv = (int32_t)pb.Hkv;
    P.N = (int32_t)pb.N;
    P.D = (int32_t)pb.D;
    P.in_bf16 = pb.dtype == RA_BF16;
    P.causal = causal ? 1 : 0;
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)pb.D));
    P.scale_log2 = sc * kLog2e;
    P.wait_limit_ns = g_wait_limit_ns;
    P.producer_delay_ns = g_producer_delay_ns;
    P.head_group = head_group(pb);
    P.err = di.err;
    P.rs = 1;
}

// The arguments take the tensor-core kernels (bf16, D in {64, 128}, 16-byte aligned bases
// and strides for the TMA maps) on an sm_103a device.
static bool tc_args(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, const ra_tensor *o,
                    const Problem &pb) {
    return pb.dtype == RA_BF16 && (pb.D == 64 || pb.D == 128) && aligned16(q) && aligned16(k) &&
           aligned16(v) && aligned16(o);
}

static bool use_tensor_cores(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                             const ra_tensor *o, const Problem &pb, const DevInfo &di) {
    return di.tc_ok && tc_args(q, k, v, o, pb);
}

// Launch the segments of one step (split into launches of <= kMaxSeg segments; all
// segments of a step have equal query length).
static ra_status run_step(StepParams &P, const Seg *segs, int nsegs, bool tc, int num_sms, int dev,
                          cudaStream_t stream) {
    const int rows_per_block = tc ? attn_tc_rows_per_block() : 16;
    for (int first = 0; first < nsegs; first += kMaxSeg) {
        const int n = std::min(nsegs - first, kMaxSeg);
        int64_t qlen = 0;
        for (int i = 0; i < n; ++i) {
            P.seg[i] = segs[first + i];
            qlen = std::max<int64_t>(qlen, segs[first + i].q1 - segs[first + i].q0);
        }
        P.nseg = (int32_t)n;
        P.rows_per_block = rows_per_block;
        P.blocks_per_seg = (int32_t)((qlen + rows_per_block - 1) / rows_per_block);
        const int64_t blocks_y = (int64_t)P.nseg * P.blocks_per_seg;
        if (blocks_y > 65535) return fail(RA_ERR_UNSUPPORTED, "too many work blocks in one step");
        P.sched = tc ? next_sched(dev) : nullptr;
        cudaError_t e = guarded_launch(tc ? "attn_tc" : "attn_simt", stream, [&] {
            return tc ? launch_attn_tc(P, (int)blocks_y, num_sms, stream) : launch_attn_simt(P, (int)blocks_y, stream);
        });
        P.chained = 1;  // later launches of this run may overlap this one's tail
        if (e != cudaSuccess) return cuda_fail(e, tc ? "attention (tensor-core) launch"
                                                     : "attention (CUDA-core) launch");
        ++t_launches;
    }
    return RA_OK;
}

// The launches of a ring run.  nfused > 0: segs holds the fused ring's segments, and one
// launch walks every step with the running result on chip (P.oacc unused).  Otherwise one
// launch per step merges into the float32 running output P.oacc (set by the caller when
// ring_size > 1); segs must hold 2 * ring_size segments.  P.rs, P.prefer_pairs and the
// common fields are the caller's.
static ra_status ring_launches(StepParams &P, bool tc, int num_sms, int dev, int64_t N, int R, int layout,
                               int causal, int nfused, Seg *segs, cudaStream_t st) {
    if (nfused > 0) {
        P.oacc = nullptr;
        P.ring_fused = 1;
        P.ring_R = R;
        P.ring_layout = layout == RA_LAYOUT_ZIGZAG ? 1 : (layout == RA_LAYOUT_STRIPED ? 2 : 0);
        P.prefer_pairs = 0;
        return run_step(P, segs, nfused, tc, num_sms, dev, st);
    }
    for (int step = 0; step < R; ++step) {
        const int n = plan_step(N, R, layout, causal, step, segs);
        if (n == 0) continue;
        ra_status s = run_step(P, segs, n, tc, num_sms, dev, st);
        if (s) return s;
    }
    return RA_OK;
}

extern "C" {

ra_status ra_attn_fwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, ra_tensor *o,
                      float *lse, int causal, float scale, void *stream) {
    return ra_ring_sim_fwd(q, k, v, o, lse, 1, RA_LAYOUT_CONTIG, causal, scale, nullptr, stream);
}

size_t ra_ring_sim_workspace_bytes(const ra_tensor *q, int ring_size) {
    if (!q || ring_size < 1) return 0;
    for (int i = 0; i < 4; ++i)
        if (q->shape[i] < 0) return 0;
    if (ring_size == 1) return 0;
    return (size_t)(q->shape[0] * q->shape[1] * q->shape[2] * q->shape[3]) * sizeof(float);
}

size_t ra_ring_sim_workspace_bytes_for(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                                       const ra_tensor *o, int ring_size, ra_layout layout, int causal) {
    Problem pb;
    if (check_qkvo(q, k, v, o, nullptr, pb, false) != RA_OK) return 0;
    if (check_ring(pb.N, ring_size, layout) != RA_OK || ring_size == 1) return 0;
    Seg segs[kMaxSeg];
    if (tc_args(q, k, v, o, pb) && fused_ring_segments(pb.N, ring_size, layout, causal, segs) > 0) return 0;
    return (size_t)(pb.B * pb.Hq * pb.N * pb.D) * sizeof(float);
}

ra_status ra_ring_sim_fwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                          ra_tensor *o, float *lse, int ring_size, ra_layout layout, int causal,
                          float scale, void *workspace, void *stream) {
    Problem pb;
    ra_status s = check_qkvo(q, k, v, o, lse, pb);
    if (s) return s;
    if (isnan(scale)) return fail(RA_ERR_INVALID_ARG, "scale is NaN");
    if ((s = check_ring(pb.N, ring_size, layout))) return s;
    if (pb.B * pb.Hq * pb.N == 0) return RA_OK;
    if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    static const char *kNeedWs =
        "workspace is NULL, and this ring run keeps a float32 running output "
        "(ra_ring_sim_workspace_bytes_for() bytes)";
    std::vector<Seg> segs(std::max(2 * (size_t)ring_size, (size_t)kMaxSeg));
    const int nfused_args =
        (ring_size > 1 && tc_args(q, k, v, o, pb)) ? fused_ring_segments(pb.N, ring_size, layout, causal, segs.data()) : 0;
    if (ring_size > 1 && nfused_args == 0 && !workspace) return fail(RA_ERR_INVALID_ARG, kNeedWs);
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    const bool tc = use_tensor_cores(q, k, v, o, pb, di);
    const int nfused = tc ? nfused_args : 0;
    if (ring_size > 1 && nfused == 0 && !workspace) return fail(RA_ERR_INVALID_ARG, kNeedWs);
    StepParams *P = new StepParams;
    fill_common(*P, q, k, v, o, lse, pb, causal, scale, di);
    P->oacc = ring_size > 1 ? static_cast<float *>(workspace) : nullptr;
    P->rs = (layout == RA_LAYOUT_STRIPED) ? ring_size : 1;
    // per-step ring launches overlap their tails with the next step's launch, so they
    // take tile-pair items; striped rings measured better with single blocks
    P->prefer_pairs = (ring_size > 1 && layout != RA_LAYOUT_STRIPED) ? 1 : 0;
    s = ring_launches(*P, tc, di.sms, di.dev, pb.N, ring_size, layout, causal, nfused, segs.data(),
                      static_cast<cudaStream_t>(stream));
    delete P;
    return s;
}

int64_t ra_ring_sim_plan(int64_t N, int ring_size, ra_layout layout, int causal, int step,
                         int64_t *segments, int64_t cap) {
    if (N < 0 || N > ((int64_t)1 << 30) || step < 0 || step >= ring_size) return -1;
    if (check_ring(N, ring_size, layout) != RA_OK) return -1;
    std::vector<Seg> segs(2 * (size_t)ring_size);
    const int n = plan_step(N, ring_size, layout, causal, step, segs.data());
    for (int64_t i = 0; i < (int64_t)n && i < cap && segments; ++i) {
        const Seg &x = segs[i];
        int64_t *o = segments + 12 * i;
        o[0] = x.q0;
        o[1] = x.q1;
        o[2] = x.k0[0];
        o[3] = x.k1[0];
        o[4] = x.k0[1];
        o[5] = x.k1[1];
        o[6] = x.flags;
        o[7] = x.rank;
        o[8] = x.q_rank;
        o[9] = x.kv_rank;
        o[10] = x.diag;
        o[11] = (layout == RA_LAYOUT_STRIPED) ? ring_size : 1;
    }
    return (int64_t)n;
}

int64_t ra_ring_sim_bwd_plan(int64_t N, int ring_size, ra_layout layout, int causal, int step, int kind,
                             int64_t *out, int64_t cap) {
    if (N < 0 || N > ((int64_t)1 << 30) || step < 0 || step >= ring_size || kind < 0 || kind > 1) return -1;
    if (check_ring(N, ring_size, layout) != RA_OK) return -1;
    const BwdPlan plan(N, ring_size, layout, causal);
    std::vector<BSeg> segs;
    plan.step(step, kind, segs);
    for (size_t i = 0; i < segs.size() && (int64_t)i < cap && out; ++i) {
        const BSeg &g = segs[i];
        const int64_t v[10] = {g.f0, g.f1, g.s0[0], g.s1[0], g.s0[1], g.s1[1], g.f_rank, g.s_rank, g.diag, g.flags};
        for (int t = 0; t < 10; ++t) out[i * 10 + t] = v[t];
    }
    return (int64_t)segs.size();
}

ra_status ra_attn_varlen_fwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                             ra_tensor *o, float *lse, const int32_t *cu_seqlens, int num_seqs,
                             int causal, float scale, void *stream) {
    Problem pb;
    ra_status s = check_qkvo(q, k, v, o, lse, pb);
    if (s) return s;
    if (isnan(scale)) return fail(RA_ERR_INVALID_ARG, "scale is NaN");
    if (pb.B > 1) return fail(RA_ERR_INVALID_ARG, "packed batches are [1, H, total, D] (B must be 1)");
    if (num_seqs < 0 || (num_seqs > 0 && !cu_seqlens))
        return fail(RA_ERR_INVALID_ARG, "cu_seqlens is NULL or num_seqs < 0");
    for (int i = 0; i < num_seqs; ++i) {
        if (cu_seqlens[i] < 0 || cu_seqlens[i + 1] < cu_seqlens[i])
            return fail(RA_ERR_INVALID_ARG, "cu_seqlens must be non-negative and non-decreasing");
    }
    if (num_seqs > 0 && cu_seqlens[num_seqs] > pb.N)
        return fail(RA_ERR_INVALID_ARG, "cu_seqlens[num_seqs] exceeds the packed length");
    if (pb.B * pb.Hq * pb.N == 0) return RA_OK;
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    StepParams *P = new StepParams;
    fill_common(*P, q, k, v, o, lse, pb, causal, scale, di);
    const bool tc = use_tensor_cores(q, k, v, o, pb, di);
    const int rows_per_block = tc ? attn_tc_rows_per_block() : 16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // one segment per non-empty sequence: its rows against its own keys only
    std::vector<Seg> segs;
    for (int i = 0; i < num_seqs; ++i) {
        const int32_t a0 = cu_seqlens[i], a1 = cu_seqlens[i + 1];
        if (a1 <= a0) continue;
        Seg g;
        memset(&g, 0, sizeof g);
        g.q0 = a0;
        g.q1 = a1;
        g.k0[0] = a0;
        g.k1[0] = a1;
        g.k0[1] = g.k1[1] = a1;
        g.flags = SEG_FIRST | SEG_FINAL;
        g.rank = i;
        segs.push_back(g);
    }
    std::stable_sort(segs.begin(), segs.end(),
                     [](const Seg &x, const Seg &y) { return x.q1 - x.q0 > y.q1 - y.q0; });
    s = RA_OK;
    for (size_t first = 0; first < segs.size() && !s; first += kMaxSeg) {
        const size_t n = std::min(segs.size() - first, (size_t)kMaxSeg);
        int64_t blocks = 0;
        for (size_t i = 0; i < n; ++i) {
            P->seg[i] = segs[first + i];
            P->seg[i].blk0 = (int32_t)blocks;
            blocks += (P->seg[i].q1 - P->seg[i].q0 + rows_per_block - 1) / rows_per_block;
        }
        P->nseg = (int32_t)n;
        P->var_blocks = 1;
        P->rows_per_block = rows_per_block;
        P->blocks_per_seg = 0;
        if (blocks > 65535) {
            s = fail(RA_ERR_UNSUPPORTED, "too many work blocks in one launch");
            break;
        }
        P->sched = tc ? next_sched(di.dev) : nullptr;
        cudaError_t e = guarded_launch(tc ? "attn_tc" : "attn_simt", st, [&] {
            return tc ? launch_attn_tc(*P, (int)blocks, di.sms, st) : launch_attn_simt(*P, (int)blocks, st);
        });
        if (e != cudaSuccess) {
            s = cuda_fail(e, "varlen attention launch");
            break;
        }
        ++t_launches;
    }
    // rows outside every sequence (padding): the identity partial, O = 0 and LSE = -inf
    int64_t covered = 0;
    std::vector<std::pair<int64_t, int64_t>> gaps;
    {
        std::vector<std::pair<int64_t, int64_t>> spans;
        for (int i = 0; i < num_seqs; ++i)
            if (cu_seqlens[i + 1] > cu_seqlens[i]) spans.push_back({cu_seqlens[i], cu_seqlens[i + 1]});
        std::sort(spans.begin(), spans.end());
        for (auto &sp : spans) {
            if (sp.first > covered) gaps.push_back({covered, sp.first});
            covered = std::max(covered, sp.second);
        }
        if (covered < pb.N) gaps.push_back({covered, pb.N});
    }
    for (size_t i = 0; i < gaps.size() && !s; ++i) {
        cudaError_t e = guarded_launch("fill_identity", st, [&] { return launch_fill_identity(o->data, pb.dtype == RA_BF16, o->stride, lse, (int)pb.B,
                                             (int)pb.Hq, (int)pb.N, (int)pb.D, (int)gaps[i].first,
                                             (int)gaps[i].second, di.sms, st); });
        if (e != cudaSuccess) s = cuda_fail(e, "padding fill launch");
        else ++t_launches;
    }
    delete P;
    return s;
}

size_t ra_attn_bwd_workspace_bytes(const ra_tensor *q) {
    if (!q) return 0;
    for (int i = 0; i < 4; ++i)
        if (q->shape[i] < 0) return 0;
    return (size_t)(q->shape[0] * q->shape[1] * q->shape[2]) * sizeof(float);
}

size_t ra_ring_sim_bwd_workspace_bytes(const ra_tensor *q, const ra_tensor *k, int ring_size) {
    if (!q || !k || ring_size < 1) return 0;
    for (int i = 0; i < 4; ++i)
        if (q->shape[i] < 0 || k->shape[i] < 0) return 0;
    const size_t rows = (size_t)(q->shape[0] * q->shape[1] * q->shape[2]);
    if (ring_size == 1) return rows * sizeof(float);
    const size_t dv_bytes = (rows * sizeof(float) + 255) & ~(size_t)255;
    const size_t nq = rows * (size_t)q->shape[3];
    const size_t nk = (size_t)(k->shape[0] * k->shape[1] * k->shape[2] * k->shape[3]);
    return dv_bytes + (nq + 2 * nk) * sizeof(float);
}

ra_status ra_ring_sim_bwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, const ra_tensor *o,
                          const float *lse, const ra_tensor *dout, ra_tensor *dq, ra_tensor *dk, ra_tensor *dv,
                          int ring_size, ra_layout layout, int causal, float scale, void *workspace,
                          void *stream) {
    Problem pb;
    ra_status s = check_qkvo(q, k, v, o, lse, pb);
    if (s) return s;
    if ((s = check_tensor(dout, "dout")) || (s = check_tensor(dq, "dq")) ||
        (s = check_tensor(dk, "dk")) || (s = check_tensor(dv, "dv")))
        return s;
    for (int i = 0; i < 4; ++i) {
        if (dout->shape[i] != q->shape[i] || dq->shape[i] != q->shape[i])
            return fail(RA_ERR_INVALID_ARG, "dout and dq must have q's shape");
        if (dk->shape[i] != k->shape[i] || dv->shape[i] != k->shape[i])
            return fail(RA_ERR_INVALID_ARG, "dk and dv must have k's shape");
    }
    if (dout->dtype != pb.dtype || dq->dtype != pb.dtype || dk->dtype != pb.dtype ||
        dv->dtype != pb.dtype)
        return fail(RA_ERR_INVALID_ARG, "gradients must share q's dtype");
    if (isnan(scale)) return fail(RA_ERR_INVALID_ARG, "scale is NaN");
    if ((s = check_ring(pb.N, ring_size, layout))) return s;
    if (pb.B * pb.Hq * pb.N == 0) return RA_OK;
    if (!workspace) return fail(RA_ERR_INVALID_ARG, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 16)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    BwdParams *Pp = new BwdParams;
    BwdParams &P = *Pp;
    memset(&P, 0, sizeof P);
    P.q = q->data;
    P.k = k->data;
    P.v = v->data;
    P.o = o->data;
    P.dout = dout->data;
    P.dq = dq->data;
    P.dk = dk->data;
    P.dv = dv->data;
    for (int i = 0; i < 3; ++i) {
        P.sq[i] = q->stride[i];
        P.sk[i] = k->stride[i];
        P.sv[i] = v->stride[i];
        P.so[i] = o->stride[i];
        P.sdo[i] = dout->stride[i];
        P.sdq[i] = dq->stride[i];
        P.sdk[i] = dk->stride[i];
        P.sdv[i] = dv->stride[i];
    }
    P.lse = lse;
    P.dvec = static_cast<float *>(workspace);
    if (ring_size > 1) {
        const size_t rows = (size_t)(pb.B * pb.Hq * pb.N);
        char *w = static_cast<char *>(workspace) + ((rows * sizeof(float) + 255) & ~(size_t)255);
        P.acc_q = reinterpret_cast<float *>(w);
        P.acc_k = P.acc_q + rows * pb.D;
        P.acc_v = P.acc_k + (size_t)(pb.B * pb.Hkv * pb.N * pb.D);
    }
    P.B = (int32_t)pb.B;
    P.Hq = (int32_t)pb.Hq;
    P.Hkv = (int32_t)pb.Hkv;
    P.N = (int32_t)pb.N;
    P.D = (int32_t)pb.D;
    P.bf16 = pb.dtype == RA_BF16;
    P.causal = causal ? 1 : 0;
    P.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)pb.D));
    P.scale_log2 = P.scale * kLog2e;
    const bool striped = layout == RA_LAYOUT_STRIPED;
    P.rs = striped ? ring_size : 1;
    P.producer_delay_ns = g_producer_delay_ns;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool tc = di.tc_ok && pb.dtype == RA_BF16 && (pb.D == 64 || pb.D == 128) && aligned16(q) &&
                    aligned16(k) && aligned16(v) && aligned16(dout) && aligned16(dq) &&
                    aligned16(dk) && aligned16(dv);
    ra_status result = RA_OK;
    cudaError_t e = guarded_launch("bwd_rowdot", st, [&] { return launch_bwd_rowdot(P, di.sms, st); });
    if (e != cudaSuccess) result = cuda_fail(e, "backward D launch");
    else ++t_launches;
    std::vector<BSeg> segs, kv_segs;
    if (result == RA_OK && tc && ring_size > 1 && fused_bwd_segments(pb.N, ring_size, layout, causal, 0, segs) &&
        fused_bwd_segments(pb.N, ring_size, layout, causal, 1, kv_segs)) {
        // one dQ launch and one dK/dV launch walk every step; gradients stay on chip
        P.ring_fused = 1;
        P.ring_R = ring_size;
        P.ring_layout = layout == RA_LAYOUT_ZIGZAG ? 1 : (layout == RA_LAYOUT_STRIPED ? 2 : 0);
        for (int kind = 0; kind < 2 && result == RA_OK; ++kind) {
            const std::vector<BSeg> &g = kind == 0 ? segs : kv_segs;
            P.nseg = (int32_t)g.size();
            P.flen = 0;
            for (size_t i = 0; i < g.size(); ++i) {
                P.seg[i] = g[i];
                P.flen = std::max<int32_t>(P.flen, g[i].f1 - g[i].f0);
            }
            P.sched = next_sched(di.dev);
            e = guarded_launch(kind == 0 ? "bwd_dq_tc" : "bwd_dkdv_tc", st, [&] {
                return launch_attn_bwd_tc(P, kind == 0 ? 1 : 2, di.sms, g_wait_limit_ns, di.err, st, kind == 1);
            });
            if (e != cudaSuccess) result = cuda_fail(e, "backward launch");
            else ++t_launches;
        }
        delete Pp;
        return result;
    }
    const BwdPlan plan(pb.N, ring_size, layout, causal);
    for (int step = 0; step < ring_size && result == RA_OK; ++step) {
        int dq_launches_this_step = 0;
        for (int kind = 0; kind < 2 && result == RA_OK; ++kind) {
            plan.step(step, kind, segs);
            for (size_t f = 0; f < segs.size() && result == RA_OK; f += kMaxBSeg) {
                const size_t n = std::min(segs.size() - f, (size_t)kMaxBSeg);
                P.nseg = (int32_t)n;
                P.flen = 0;
                for (size_t i = 0; i < n; ++i) {
                    P.seg[i] = segs[f + i];
                    P.flen = std::max<int32_t>(P.flen, segs[f + i].f1 - segs[f + i].f0);
                }
                const int parts = kind == 0 ? 1 : 2;
                // a step's dK/dV launch follows its dQ launch directly, unless the dQ
                // segments took several launches
                const bool after_dq = kind == 1 && f == 0 && dq_launches_this_step == 1;
                P.sched = tc ? next_sched(di.dev) : nullptr;
                e = guarded_launch(tc ? (kind == 0 ? "bwd_dq_tc" : "bwd_dkdv_tc") : (kind == 0 ? "bwd_dq_simt" : "bwd_dkdv_simt"),
                                   st, [&] {
                                       return tc ? launch_attn_bwd_tc(P, parts, di.sms, g_wait_limit_ns, di.err, st, after_dq)
                                                 : launch_attn_bwd_simt(P, parts, st);
                                   });
                if (kind == 0) ++dq_launches_this_step;
                if (e != cudaSuccess) result = cuda_fail(e, "backward launch");
                else ++t_launches;
            }
        }
    }
    delete Pp;
    return result;
}

ra_status ra_attn_bwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, const ra_tensor *o,
                      const float *lse, const ra_tensor *dout, ra_tensor *dq, ra_tensor *dk,
                      ra_tensor *dv, int causal, float scale, void *workspace, void *stream) {
    return ra_ring_sim_bwd(q, k, v, o, lse, dout, dq, dk, dv, 1, RA_LAYOUT_CONTIG, causal, scale, workspace,
                           stream);
}

// ---------------------------------------------------------------- host-buffer entry point

// Boundaries (in KV heads) of the host-buffer call's ng head groups: kb[0] = 0 < kb[1] < ...
// < kb[ng] = hkv.  Copy-bound with heads to spare (hkv >= 3 ng, ng >= 4): sizes falling in
// proportion to ng, ng - 1, ..., 1 (to one head for 32 heads in 8 groups), so that what
// nothing overlaps at the end - the last groups' kernels and copies out, after the last copy
// in - is small; else equal groups.
static void host_group_bounds(int64_t hkv, int ng, bool copy_bound, int64_t *kb) {
    const bool falling = copy_bound && ng >= 4 && hkv >= 3 * (int64_t)ng;
    const int64_t wsum = (int64_t)ng * (ng + 1) / 2;
    kb[0] = 0;
    for (int g = 1; g <= ng; ++g) {
        const int64_t w = (int64_t)g * ng - (int64_t)g * (g - 1) / 2;  // weights ng, ng-1, ... of groups < g
        int64_t b = falling ? (hkv * w + wsum / 2) / wsum : hkv * g / ng;
        b = std::max<int64_t>(b, kb[g - 1] + 1);
        b = std::min<int64_t>(b, hkv - (ng - g));
        kb[g] = b;
    }
}

extern "C" int ra_debug_host_group_bounds(int64_t hkv, int ng, int copy_bound, int64_t *out) {
    if (hkv < 1 || ng < 1 || ng > kHostGroups || ng > hkv || !out) return -1;
    host_group_bounds(hkv, ng, copy_bound != 0, out);
    return ng;
}

// Streams and events of the host-buffer pipeline, created once per device (copies in on
// one stream, copies out on another, so both directions of the link run at once).
struct HostPipe {
    cudaStream_t cin = nullptr, cout = nullptr;
    cudaEvent_t ev[2 * kHostGroups + 2] = {};
    bool ready = false;
};
static HostPipe g_pipe[kMaxDev];
static std::mutex g_pipe_mu;

static bool host_pipe(int dev, HostPipe *&hp, std::string &msg) {
    if (dev < 0 || dev >= kMaxDev) {
        msg = "device ordinal out of range";
        return false;
    }
    hp = &g_pipe[dev];
    if (hp->ready) return true;
    cudaError_t e = cudaStreamCreateWithFlags(&hp->cin, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->cout, cudaStreamNonBlocking);
    for (int i = 0; e == cudaSuccess && i < 2 * kHostGroups + 2; ++i)
        e = cudaEventCreateWithFlags(&hp->ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        msg = std::string("host pipeline set-up: ") + cudaGetErrorString(e);
        return false;
    }
    hp->ready = true;
    return true;
}

static bool host_contiguous(const ra_tensor *t) {
    return t->stride[3] == 1 && t->stride[2] == t->shape[3] && t->stride[1] == t->shape[2] * t->shape[3] &&
           t->stride[0] == t->shape[1] * t->shape[2] * t->shape[3];
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t ra_ring_sim_fwd_host_workspace_bytes(const ra_tensor *q, const ra_tensor *k, int ring_size) {
    if (!q || !k || ring_size < 1 || !is_dtype(q->dtype)) return 0;
    for (int i = 0; i < 4; ++i)
        if (q->shape[i] < 0 || k->shape[i] < 0) return 0;
    const size_t es = (size_t)esize(q->dtype);
    const size_t nq = (size_t)(q->shape[0] * q->shape[1] * q->shape[2] * q->shape[3]);
    const size_t nk = (size_t)(k->shape[0] * k->shape[1] * k->shape[2] * k->shape[3]);
    const size_t rows = (size_t)(q->shape[0] * q->shape[1] * q->shape[2]);
    // device q, o, k, v, lse, and the ring's running result for one head group at most
    // (every group runs on the caller's stream in turn)
    return 2 * align256(nq * es) + 2 * align256(nk * es) + align256(rows * sizeof(float)) +
           (ring_size > 1 ? align256(nq * sizeof(float)) : 0);
}

ra_status ra_ring_sim_fwd_host(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, ra_tensor *o,
                               float *lse, int ring_size, ra_layout layout, int causal, float scale,
                               void *workspace, size_t workspace_bytes, void *stream) {
    Problem pb;
    ra_status s = check_qkvo(q, k, v, o, lse, pb);
    if (s) return s;
    if (isnan(scale)) return fail(RA_ERR_INVALID_ARG, "scale is NaN");
    if ((s = check_ring(pb.N, ring_size, layout))) return s;
    if (!host_contiguous(q) || !host_contiguous(k) || !host_contiguous(v) || !host_contiguous(o))
        return fail(RA_ERR_INVALID_ARG, "host tensors must be contiguous [B, H, N, D]");
    if (pb.B * pb.Hq * pb.N == 0) return RA_OK;
    const size_t need = ra_ring_sim_fwd_host_workspace_bytes(q, k, ring_size);
    if (!workspace || workspace_bytes < need)
        return fail(RA_ERR_INVALID_ARG, "workspace is NULL or smaller than ra_ring_sim_fwd_host_workspace_bytes()");
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe *hp = nullptr;
    if (!host_pipe(di.dev, hp, msg)) return fail(RA_ERR_CUDA, msg);
    const int64_t B = pb.B, Hq = pb.Hq, Hkv = pb.Hkv, N = pb.N, D = pb.D, G = Hq / Hkv;
    const size_t es = (size_t)esize(pb.dtype);
    const size_t nq = (size_t)(B * Hq * N * D), nk = (size_t)(B * Hkv * N * D);
    char *w = static_cast<char *>(workspace);
    char *dq = w, *dout = dq + align256(nq * es), *dk = dout + align256(nq * es), *dv = dk + align256(nk * es);
    float *dl = reinterpret_cast<float *>(dv + align256(nk * es));
    void *ring_ws = ring_size > 1 ? static_cast<void *>(reinterpret_cast<char *>(dl) + align256((size_t)(B * Hq * N) * 4))
                                  : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Head groups of whole KV heads (with their G query heads each), every batch in one
    // launch.  More groups overlap more of the copies with the kernels, and the last
    // group's kernel and copy out, which nothing overlaps, get shorter; but each group's
    // launch must still fill the persistent grid: at least two rounds of 256-row blocks
    // where that leaves two or more groups (one KV head of the 8-rank N = 32K ring is a
    // single round of 128 blocks, and eight such groups ran at a third of the grid's
    // rate).  When the copies take much longer than the kernels (the dense 4K workload
    // moves 269 MB for 0.3 TFLOP), the kernels hide behind them whatever their grid fill;
    // eight groups then beat sixteen (the copies alone, measured on a GB300: 1.16 ms
    // against 1.22 ms for that workload's 269 MB).  (Rates: ~1.2 PFLOP/s for the kernels,
    // ~200 GB/s each way for pinned host copies.)
    const double flops = 4.0 * (double)(B * Hq) * (double)N * (double)N * (double)D * (causal ? 0.5 : 1.0);
    const double bytes = (double)(2 * nq + 2 * nk) * (double)es;
    const bool copy_bound = flops / 1.2e15 < 0.5 * bytes / 2.0e11;
    const int64_t blocks = B * Hq * ((N + 255) / 256);  // work blocks of the whole problem
    const int64_t most = std::min<int64_t>(Hkv, kHostGroups);
    const int ng = (int)(copy_bound ? most : std::min<int64_t>(most, std::max<int64_t>(2, blocks / (2 * (int64_t)di.sms))));
    cudaError_t e = cudaEventRecord(hp->ev[2 * kHostGroups], st);  // prior work on the caller's stream
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->cin, hp->ev[2 * kHostGroups], 0);
    const size_t qrow = (size_t)(N * D) * es;  // bytes of one head's rows
    int64_t kb[kHostGroups + 1];
    host_group_bounds(Hkv, ng, copy_bound, kb);
    for (int g = 0; g < ng && e == cudaSuccess; ++g) {
        const int64_t k0 = kb[g], k1 = kb[g + 1], q0 = k0 * G, q1 = k1 * G;
        // in: q, k, v rows of the group, every batch (one 2-D copy each)
        e = cudaMemcpy2DAsync(dq + q0 * qrow, (size_t)Hq * qrow, static_cast<const char *>(q->data) + q0 * qrow,
                              (size_t)Hq * qrow, (size_t)(q1 - q0) * qrow, (size_t)B, cudaMemcpyHostToDevice, hp->cin);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(dk + k0 * qrow, (size_t)Hkv * qrow, static_cast<const char *>(k->data) + k0 * qrow,
                                  (size_t)Hkv * qrow, (size_t)(k1 - k0) * qrow, (size_t)B, cudaMemcpyHostToDevice,
                                  hp->cin);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(dv + k0 * qrow, (size_t)Hkv * qrow, static_cast<const char *>(v->data) + k0 * qrow,
                                  (size_t)Hkv * qrow, (size_t)(k1 - k0) * qrow, (size_t)B, cudaMemcpyHostToDevice,
                                  hp->cin);
        if (e == cudaSuccess) e = cudaEventRecord(hp->ev[g], hp->cin);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->ev[g], 0);
        if (e != cudaSuccess) break;
        // compute: the group's heads of every batch, viewed inside the full device tensors;
        // their LSE goes to a packed [B, group heads, N] slice of the LSE buffer (the
        // group's rows of the full [B, Hq, N] layout are strided across batches)
        ra_tensor tq = *q, tk = *k, tv = *v, to = *o;
        const int64_t sq[4] = {Hq * N * D, N * D, D, 1}, sk[4] = {Hkv * N * D, N * D, D, 1};
        for (int i = 0; i < 4; ++i) {
            tq.stride[i] = to.stride[i] = sq[i];
            tk.stride[i] = tv.stride[i] = sk[i];
        }
        tq.shape[1] = to.shape[1] = q1 - q0;
        tk.shape[1] = tv.shape[1] = k1 - k0;
        tq.data = dq + q0 * qrow;
        to.data = dout + q0 * qrow;
        tk.data = dk + k0 * qrow;
        tv.data = dv + k0 * qrow;
        float *glse = dl + B * q0 * N;
        s = ra_ring_sim_fwd(&tq, &tk, &tv, &to, glse, ring_size, layout, causal, scale, ring_ws, stream);
        if (s != RA_OK) return s;
        e = cudaEventRecord(hp->ev[kHostGroups + g], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->cout, hp->ev[kHostGroups + g], 0);
        // out: o rows and LSE of the group
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(static_cast<char *>(o->data) + q0 * qrow, (size_t)Hq * qrow, dout + q0 * qrow,
                                  (size_t)Hq * qrow, (size_t)(q1 - q0) * qrow, (size_t)B, cudaMemcpyDeviceToHost, hp->cout);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(lse + q0 * N, (size_t)(Hq * N) * 4, dl + B * q0 * N, (size_t)((q1 - q0) * N) * 4,
                                  (size_t)((q1 - q0) * N) * 4, (size_t)B, cudaMemcpyDeviceToHost, hp->cout);
    }
    // the caller's stream sees every copy out complete
    if (e == cudaSuccess) e = cudaEventRecord(hp->ev[2 * kHostGroups + 1], hp->cout);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->ev[2 * kHostGroups + 1], 0);
    if (e != cudaSuccess) return cuda_fail(e, "host-buffer pipeline");
    return RA_OK;
}

ra_status ra_ulysses_all_to_all(const ra_tensor *in, ra_tensor *out, int sp, int to_heads,
                                void *stream) {
    ra_status s;
    if ((s = check_tensor(in, "in")) || (s = check_tensor(out, "out"))) return s;
    if (in->dtype != out->dtype) return fail(RA_ERR_INVALID_ARG, "in and out must share a dtype");
    if (sp < 1) return fail(RA_ERR_INVALID_ARG, "sp must be >= 1");
    const ra_tensor *seq = to_heads ? in : out;
    const ra_tensor *head = to_heads ? out : in;
    const int64_t S = seq->shape[1] * sp, H = seq->shape[2], D = seq->shape[3];
    if (seq->shape[0] != sp || head->shape[0] != sp || head->shape[1] != S ||
        head->shape[2] * sp != H || head->shape[3] != D || H % sp != 0)
        return fail(RA_ERR_INVALID_ARG,
                    "expected sequence shards [sp, S/sp, H, D] and head shards [sp, S, H/sp, D]");
    if (S * H * D == 0) return RA_OK;
    if (S > INT32_MAX || H > INT32_MAX || D > INT32_MAX)
        return fail(RA_ERR_UNSUPPORTED, "dimension too large");
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    UlyssesParams P;
    memset(&P, 0, sizeof P);
    P.in = in->data;
    P.out = out->data;
    for (int i = 0; i < 4; ++i) {
        P.si[i] = in->stride[i];
        P.so[i] = out->stride[i];
    }
    P.sp = sp;
    P.S = (int32_t)S;
    P.H = (int32_t)H;
    P.D = (int32_t)D;
    P.esize = esize(in->dtype);
    P.to_heads = to_heads ? 1 : 0;
    const int64_t per16 = 16 / P.esize;
    P.vec = (D % per16 == 0) && aligned16(in) && aligned16(out);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = guarded_launch("ulysses", st, [&] { return launch_ulysses(P, di.sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "ulysses launch");
    ++t_launches;
    return RA_OK;
}

ra_status ra_lse_merge(ra_tensor *o_acc, float *lse_acc, const ra_tensor *o_blk,
                       const float *lse_blk, void *stream) {
    ra_status s;
    if ((s = check_tensor(o_acc, "o_acc")) || (s = check_tensor(o_blk, "o_blk"))) return s;
    if (o_acc->dtype != RA_F32) return fail(RA_ERR_INVALID_ARG, "o_acc must be float32");
    for (int i = 0; i < 4; ++i)
        if (o_acc->shape[i] != o_blk->shape[i])
            return fail(RA_ERR_INVALID_ARG, "o_acc and o_blk shapes differ");
    const int64_t rows = o_acc->shape[0] * o_acc->shape[1] * o_acc->shape[2];
    if (rows == 0 || o_acc->shape[3] == 0) return RA_OK;
    if (!lse_acc || !lse_blk) return fail(RA_ERR_INVALID_ARG, "lse pointer is NULL");
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    MergeParams P;
    memset(&P, 0, sizeof P);
    P.oacc = static_cast<float *>(o_acc->data);
    P.lse_acc = lse_acc;
    P.oblk = o_blk->data;
    P.lse_blk = lse_blk;
    for (int i = 0; i < 3; ++i) {
        P.sa[i] = o_acc->stride[i];
        P.sb[i] = o_blk->stride[i];
    }
    P.blk_bf16 = o_blk->dtype == RA_BF16;
    P.H = (int32_t)o_acc->shape[1];
    P.N = (int32_t)o_acc->shape[2];
    P.D = (int32_t)o_acc->shape[3];
    P.rows = rows;
    const int64_t bvec = P.blk_bf16 ? 4 : 4;  // elements per vector access
    const uintptr_t balign = P.blk_bf16 ? 8 : 16;
    P.vec = (P.D % 4 == 0) && reinterpret_cast<uintptr_t>(P.oacc) % 16 == 0 &&
            reinterpret_cast<uintptr_t>(P.oblk) % balign == 0 && P.sa[0] % 4 == 0 &&
            P.sa[1] % 4 == 0 && P.sa[2] % 4 == 0 && P.sb[0] % bvec == 0 && P.sb[1] % bvec == 0 &&
            P.sb[2] % bvec == 0;
    // half a warp per row moves 8 values per lane: 16-byte block rows for bf16 too
    P.half_warp = P.vec && P.D <= 128 &&
                  (!P.blk_bf16 || (reinterpret_cast<uintptr_t>(P.oblk) % 16 == 0 && P.sb[0] % 8 == 0 &&
                                   P.sb[1] % 8 == 0 && P.sb[2] % 8 == 0));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = guarded_launch("lse_merge", st, [&] { return launch_lse_merge(P, di.sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "lse_merge launch");
    ++t_launches;
    return RA_OK;
}

ra_status ra_check_device_error(void *stream) {
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int word = 0;
    e = cudaMemcpy(&word, di.err, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpy(di.err, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
        if (word == DERR_TIMEOUT)
            return fail(RA_ERR_TIMEOUT, "a device pipeline wait exceeded its time limit");
        if (word == DERR_BOUNDS)
            return fail(RA_ERR_BOUNDS, "a device-side bounds check failed (the access was skipped)");
        return fail(RA_ERR_CUDA, "device error word " + std::to_string(word));
    }
    return RA_OK;
}

void ra_debug_set_wait_limit_ns(int64_t ns) { g_wait_limit_ns = ns < 0 ? 2000000000LL : ns; }

void ra_debug_set_producer_delay_ns(int64_t ns) { g_producer_delay_ns = ns < 0 ? 0 : std::min<int64_t>(ns, 100000000LL); }

void ra_debug_fail_next_launches(int n) { t_inject_launch_failures = n > 0 ? n : 0; }

void ra_debug_time_launches(int enable) { t_time_launches = enable != 0; }

int ra_debug_launch_times(float *ms, int cap, char *names, int name_len) {
    const int n = (int)t_timed.size();
    for (int i = 0; i < n; ++i) {
        TimedLaunch &t = t_timed[i];
        float v = -1.f;
        if (cudaEventSynchronize(t.stop) == cudaSuccess && cudaEventElapsedTime(&v, t.start, t.stop) != cudaSuccess)
            v = -1.f;
        if (i < cap) {
            if (ms) ms[i] = v;
            if (names && name_len > 0) {
                strncpy(names + (size_t)i * name_len, t.name, (size_t)name_len - 1);
                names[(size_t)i * name_len + name_len - 1] = 0;
            }
        }
        cudaEventDestroy(t.start);
        cudaEventDestroy(t.stop);
    }
    t_timed.clear();
    cudaGetLastError();
    return n;
}

int ra_debug_bounds_checked(void) {
#ifdef RA_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

ra_status ra_debug_bounds_selftest(void *stream) {
    if (!ra_debug_bounds_checked())
        return fail(RA_ERR_UNSUPPORTED, "this library was built without device bounds checks");
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    cudaError_t e = launch_bounds_selftest(di.err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bounds self-test launch");
    ++t_launches;
    return RA_OK;
}

ra_status ra_debug_wait_selftest(int64_t limit_ns, void *stream) {
    if (limit_ns < 0 || limit_ns > 10000000000LL)
        return fail(RA_ERR_INVALID_ARG, "limit_ns must be in [0, 1e10]");
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    cudaError_t e = launch_wait_selftest(limit_ns, di.err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
    ++t_launches;
    return RA_OK;
}

int ra_debug_work_counters_in_use(void *stream) {
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return -1;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
    static int host[2 * kSchedSlots];
    std::lock_guard<std::mutex> lk(g_mu);
    if (cudaMemcpyFromSymbol(host, g_sched, sizeof(host)) != cudaSuccess) return -1;
    int n = 0;
    for (int i = 0; i < kSchedSlots; ++i) n += (host[2 * i] != 0 || host[2 * i + 1] != 0);
    return n;
}

const char *ra_last_error(void) { return t_last_error.c_str(); }

int64_t ra_launch_count(int reset) {
    const int64_t n = t_launches;
    if (reset) t_launches = 0;
    return n;
}

int ra_version(void) { return 100; }

}  // extern "C"

// ---------------------------------------------------------------- allocation-free ring run
//
// Some callers cannot let this library allocate device memory: a framework whose own
// memory pool owns the device, a latency-critical loop where cudaMalloc/cudaFree would
// synchronise the device, or a host application that hands a plugin only its input and
// output buffers.  ra_ring_sim_fwd_noalloc serves them with the schedule of
// ra_ring_sim_fwd: the fused ring keeps its running result on chip and needs no scratch;
// the per-step launches keep the float32 running output, which ra_ring_sim_fwd holds in a
// caller-provided workspace, in the fixed array below.  The call allocates nothing (no
// cudaMalloc/cudaFree, no host heap on success).
//
// The array is part of this module: every GPU that loads the library holds it until the
// process exits.  Host code must not pass the array's name to a kernel (in host code it
// is only a stand-in for the device symbol); the kernels get its device address, looked
// up once per device with that device current.

namespace {

constexpr int64_t kNoAllocScratchFloats = (int64_t)8 << 20;  // 8 Mi floats = 32 MiB
constexpr int kNoAllocMaxRing = kMaxSeg / 2;                  // one launch per ring step
constexpr int kNoAllocMaxSeg = 2 * kNoAllocMaxRing;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

static float *g_noalloc_ptr[kMaxDev];

// Set-up, once per device, with that device current: the scratch array's device address.
static bool noalloc_scratch(int dev, float **out, std::string &msg) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            msg = std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e);
            return false;
        }
        g_noalloc_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return true;
}

}  // namespace

extern "C" ra_status ra_ring_sim_fwd_noalloc(const ra_tensor *q, const ra_tensor *k,
                                             const ra_tensor *v, ra_tensor *o, float *lse,
                                             int ring_size, ra_layout layout, int causal,
                                             float scale, void *stream) {
    Problem pb;
    ra_status s = check_qkvo(q, k, v, o, lse, pb);
    if (s) return s;
    if (isnan(scale)) return fail(RA_ERR_INVALID_ARG, "scale is NaN");
    if ((s = check_ring(pb.N, ring_size, layout))) return s;
    if (pb.B * pb.Hq * pb.N == 0) return RA_OK;
    DevInfo di;
    std::string msg;
    if (!device_info(di, msg)) return fail(RA_ERR_CUDA, msg);
    const bool tc = use_tensor_cores(q, k, v, o, pb, di);
    // the schedule of ra_ring_sim_fwd, in a fixed array: the fused ring (running result on
    // chip, no scratch) when it applies, else one launch per step over the scratch array
    Seg segs[kNoAllocMaxSeg];
    const int nfused = (tc && ring_size > 1) ? fused_ring_segments(pb.N, ring_size, layout, causal, segs) : 0;
    float *scratch = nullptr;
    if (ring_size > 1 && nfused == 0) {
        if (ring_size > kNoAllocMaxRing)
            return fail(RA_ERR_UNSUPPORTED,
                        "ra_ring_sim_fwd_noalloc: ring_size above 64 outside the fused ring");
        if (pb.B * pb.Hq * pb.N * pb.D > kNoAllocScratchFloats)
            return fail(RA_ERR_UNSUPPORTED,
                        "ra_ring_sim_fwd_noalloc: B*Hq*N*D exceeds its fixed scratch of 8Mi floats "
                        "(32 MiB); use ra_ring_sim_fwd with a caller-provided workspace");
        if (!noalloc_scratch(di.dev, &scratch, msg)) return fail(RA_ERR_CUDA, msg);
    }
    StepParams P;
    fill_common(P, q, k, v, o, lse, pb, causal, scale, di);
    P.oacc = scratch;
    P.rs = (layout == RA_LAYOUT_STRIPED) ? ring_size : 1;
    P.prefer_pairs = (ring_size > 1 && layout != RA_LAYOUT_STRIPED) ? 1 : 0;
    return ring_launches(P, tc, di.sms, di.dev, pb.N, ring_size, layout, causal, nfused, segs,
                         static_cast<cudaStream_t>(stream));
}
