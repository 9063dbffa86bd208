// Host side of the MTTKRP library: the C ABI of include/mttkrp.h, the planner
// (mode classification, inner-group choice, tiles, split counts, workspace
// layout) and the launch sequence of one mode:
//   1. factor-product tables G (pre modes, with Y base offsets) and, for an
//      inner group of several modes, Binner;
//   2. the main kernel (SIMT or tensor-core path) over tiles x split ranges;
//   3. if the contraction range was split, the fixed-order fp64 reduction.
// Everything is enqueued on the caller's stream; nothing synchronises.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "internal.h"
#include "tc.h"

namespace mk {
namespace {

thread_local char g_errmsg[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_errmsg, sizeof(g_errmsg), fmt, ap);
    va_end(ap);
    return code;
}

constexpr int64_t kMaxR = 65536;
constexpr int64_t kMaxNumel = (int64_t)1 << 40;
// Inner-group size the planner aims for (at least this many j values per pi),
// as long as at least kMinPre pre indices remain to spread over split ranges.
constexpr int64_t kInnerMin = 64;
constexpr int64_t kMinPre = 64;
// Longest fp32 accumulation chain (in products) allowed in one SIMT thread; more
// contraction work is split into ranges whose partials are summed in fp64.
constexpr int64_t kSimtChain = 8192;
// CTAs the SIMT grid aims for: 2 waves of 2 CTAs on each of 152 SMs.
constexpr int64_t kSimtTargetCtas = 608;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

void classify(const Plan& p, int k, ModeGeom& g) {
    const int d = p.d;
    g.k = k;
    g.I = p.dims[k];
    g.R = p.R;
    g.s_k = p.strides[k];
    int64_t Q = 1;
    for (int n = k + 1; n < d; ++n) Q *= p.dims[n];
    bool in_group[kMaxD] = {false};
    int64_t J = 1, Jq = 1;
    const int64_t others = [&] {
        int64_t x = 1;
        for (int n = 0; n < d; ++n)
            if (n != k) x *= p.dims[n];
        return x;
    }();
    // grow the group by one more mode only while it is small and enough pre
    // indices would remain afterwards (the first mode is always taken)
    auto grow = [&](int64_t J_now, int64_t dim) {
        return J_now == 1 || (J_now < kInnerMin && others / (J_now * dim) >= kMinPre);
    };
    if (Q >= kInnerMin) {
        // trailing modes after k
        for (int n = d - 1; n > k && grow(J, p.dims[n]); --n) {
            in_group[n] = true;
            J *= p.dims[n];
        }
        Jq = J;
    } else {
        // all modes after k, then the last modes before k
        for (int n = k + 1; n < d; ++n) in_group[n] = true;
        J = Jq = Q;
        for (int n = k - 1; n >= 0 && grow(J, p.dims[n]); --n) {
            in_group[n] = true;
            J *= p.dims[n];
        }
    }
    g.J = J;
    g.Jq = Jq;
    g.IQ = (k > 0) ? p.strides[k - 1] : 0;
    g.ngroup = 0;
    g.npm = 0;
    g.npre = 1;
    for (int n = 0; n < d; ++n) {
        if (n == k) continue;
        if (in_group[n]) {
            g.group[g.ngroup++] = n;
        } else {
            g.pm[g.npm++] = n;
            g.npre *= p.dims[n];
        }
    }
}

// The matrix-based variant: every mode but k forms the inner group, so the B
// operand is the whole Khatri-Rao product (J = prod_{n != k} I_n rows), with
// one pre index.
void classify_explicit(const Plan& p, int k, ModeGeom& g) {
    g.k = k;
    g.I = p.dims[k];
    g.R = p.R;
    g.s_k = p.strides[k];
    g.J = 1;
    g.Jq = 1;
    for (int n = 0; n < p.d; ++n) {
        if (n == k) continue;
        g.J *= p.dims[n];
        if (n > k) g.Jq *= p.dims[n];
    }
    g.IQ = (k > 0) ? p.strides[k - 1] : 0;
    g.ngroup = 0;
    g.npm = 0;
    g.npre = 1;
    for (int n = 0; n < p.d; ++n)
        if (n != k) g.group[g.ngroup++] = n;
}

void plan_simt(ModePlan& mp) {
    const ModeGeom& g = mp.g;
    mp.path = MTTKRP_PATH_SIMT;
    mp.bn = g.R > 64 ? 128 : 64;
    mp.bm = g.I >= 96 ? 128 : (g.I > 32 ? 64 : 32);
    const int64_t tiles = cdiv(g.I, mp.bm) * cdiv(g.R, mp.bn);
    const int64_t K = g.npre * g.J;
    int64_t S = cdiv(K, kSimtChain);
    const int64_t s_par = cdiv(kSimtTargetCtas, tiles);
    if (s_par > S) S = s_par;
    if (S > g.npre) S = g.npre;
    if (S > 65535) S = 65535;
    if (S < 1) S = 1;
    mp.pre_per_split = cdiv(g.npre, S);
    mp.splits = cdiv(g.npre, mp.pre_per_split);
}

void layout_workspace(const Plan& p, ModePlan& mp) {
    const ModeGeom& g = mp.g;
    size_t off = 256;  // first 256 bytes reserved
    mp.off_partials = off;
    if (mp.splits > 1) off = align256(off + (size_t)mp.splits * g.I * g.R * sizeof(float));
    mp.off_binner = off;
    if (mp.path == MTTKRP_PATH_TC) {
        off = align256(off + tc_binner_bytes(mp));
    } else if (g.ngroup > 1) {
        off = align256(off + (size_t)g.J * g.R * sizeof(float));
    }
    mp.off_gtab = off;
    off = align256(off + (size_t)g.npre * g.R * sizeof(float));
    mp.off_base = off;
    off = align256(off + (size_t)g.npre * sizeof(int64_t));
    mp.off_t1 = off;
    if (mp.explicit_krp) {
        // product of the group's factors but the last: J / I_last rows of R
        const int64_t rows = g.J / p.dims[g.group[g.ngroup - 1]];
        off = align256(off + (size_t)rows * g.R * sizeof(float));
    }
    mp.off_end = off;
    mp.total = off;
}

// Plan-level workspace regions after every mode's own needs, shared by all
// modes of a call: for fp16-split modes the largest |Y| of every slab of mode 0
// (one slab when some fp16-split mode sums over mode 0 inside its tensor-memory
// accumulation, i.e. has it in its inner group), then the fp16 images of Y
// (tc_img modes) written for the first such mode of a call.
void place_plan_regions(Plan& p) {
    size_t base = 0;
    p.img_nat = p.img_t = 0;
    p.fuse_mode = -1;
    bool fp16 = false, slab_ok = true;
    for (int k = 0; k < p.d; ++k) {
        const ModePlan& mp = p.mode[k];
        if (mp.path == MTTKRP_PATH_TC && (mp.tc_img || mp.tc_h2)) {
            fp16 = true;
            if (k != 0 && !(mp.g.npm > 0 && mp.g.pm[0] == 0)) slab_ok = false;
            if (mp.tc_img) {
                if (mp.tc_img_t)
                    p.img_t = 1;
                else
                    p.img_nat = 1;
            }
        }
        if (mp.total > base) base = mp.total;
    }
    p.slab_on = (fp16 && slab_ok && p.dims[0] > 1) ? 1 : 0;
    p.nslab = p.slab_on ? p.dims[0] : 1;
    p.off_slab = 0;
    if (!fp16) return;
    base = align256(base);
    p.off_slab = base;
    base = align256(base + (size_t)(p.nslab + 1) * sizeof(uint32_t));   // + the image pass's out-of-range flag
    int64_t numel = 1;
    for (int n = 0; n < p.d; ++n) numel *= p.dims[n];
    const size_t img = 2 * align256((size_t)numel * 2);   // hi and lo, 2 bytes an element
    const size_t off_nat = base;
    const size_t off_t = base + (p.img_nat ? img : 0);
    const size_t total = off_t + (p.img_t ? img : 0);
    for (int k = 0; k < p.d; ++k) {
        ModePlan& mp = p.mode[k];
        if (mp.path != MTTKRP_PATH_TC || !(mp.tc_img || mp.tc_h2)) continue;
        mp.off_img = off_nat;
        mp.off_timg = off_t;
        mp.total = total;
    }
    p.fuse_mode = tc_pick_fuse_mode(p);
}

int plan_mode(Plan& p, int k, int path) {
    ModePlan& mp = p.mode[k];
    memset(&mp, 0, sizeof(mp));
    classify(p, k, mp.g);
    // MTTKRP_PATH_TC_TF32: the tensor-core kernels without the fp16 split
    const bool allow_fp16 = path != MTTKRP_PATH_TC_TF32;
    if (path == MTTKRP_PATH_TC_TF32) path = MTTKRP_PATH_TC;
    if (path == MTTKRP_PATH_TC_EXPLICIT_KRP) {
        // the matrix-based variant: tensor-core kernels over the explicit
        // Khatri-Rao product; a misaligned Y runs the matrix-free SIMT plan
        ModePlan& alt = p.simt_alt[k];
        alt = mp;
        plan_simt(alt);
        layout_workspace(p, alt);
        classify_explicit(p, k, mp.g);
        mp.explicit_krp = 1;
        if (!tc_plan(p, mp, true)) return MTTKRP_ERR_UNSUPPORTED;
        layout_workspace(p, mp);
        if (cdiv(alt.g.I, alt.bm) <= 65535 && alt.total > mp.total) mp.total = alt.total;
        return MTTKRP_OK;
    }
    if (path == MTTKRP_PATH_AUTO) {
        path = MTTKRP_PATH_SIMT;
        if (tc_prefer(mp)) {
            ModePlan trial = mp;
            if (tc_plan(p, trial, true)) path = MTTKRP_PATH_TC;
        }
    }
    ModePlan& alt = p.simt_alt[k];
    alt = mp;
    plan_simt(alt);
    layout_workspace(p, alt);
    const bool simt_ok = cdiv(alt.g.I, alt.bm) <= 65535;  // row tiles run along gridDim.y
    if (path == MTTKRP_PATH_TC) {
        if (!tc_plan(p, mp, allow_fp16)) return MTTKRP_ERR_UNSUPPORTED;
        layout_workspace(p, mp);
        if (simt_ok && alt.total > mp.total) mp.total = alt.total;
    } else {
        if (!simt_ok) return MTTKRP_ERR_UNSUPPORTED;
        mp = alt;
    }
    return MTTKRP_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

// Event pair for the next timed main kernel of mode k (grown on demand).
cudaError_t timing_pair(Plan& p, int k, cudaEvent_t* e0, cudaEvent_t* e1) {
    if (p.ev_n[k] == p.ev_cap[k]) {
        const int cap = p.ev_cap[k] ? 2 * p.ev_cap[k] : 64;
        cudaEvent_t* s = new (std::nothrow) cudaEvent_t[cap];
        cudaEvent_t* t = new (std::nothrow) cudaEvent_t[cap];
        if (!s || !t) {
            delete[] s;
            delete[] t;
            return cudaErrorMemoryAllocation;
        }
        for (int i = 0; i < p.ev_cap[k]; ++i) {
            s[i] = p.ev_start[k][i];
            t[i] = p.ev_stop[k][i];
        }
        for (int i = p.ev_cap[k]; i < cap; ++i) s[i] = t[i] = nullptr;
        delete[] p.ev_start[k];
        delete[] p.ev_stop[k];
        p.ev_start[k] = s;
        p.ev_stop[k] = t;
        p.ev_cap[k] = cap;
    }
    const int i = p.ev_n[k];
    cudaError_t err;
    if (p.ev_start[k][i] == nullptr && (err = cudaEventCreate(&p.ev_start[k][i])) != cudaSuccess) return err;
    if (p.ev_stop[k][i] == nullptr && (err = cudaEventCreate(&p.ev_stop[k][i])) != cudaSuccess) return err;
    *e0 = p.ev_start[k][i];
    *e1 = p.ev_stop[k][i];
    return cudaSuccess;
}

void free_events(Plan& p) {
    for (int k = 0; k < kMaxD; ++k) {
        for (int i = 0; i < p.ev_cap[k]; ++i) {
            if (p.ev_start[k][i]) cudaEventDestroy(p.ev_start[k][i]);
            if (p.ev_stop[k][i]) cudaEventDestroy(p.ev_stop[k][i]);
        }
        delete[] p.ev_start[k];
        delete[] p.ev_stop[k];
        p.ev_start[k] = p.ev_stop[k] = nullptr;
        p.ev_cap[k] = p.ev_n[k] = 0;
    }
}

int run_mode(Plan& p, const float* Y, const float* const* factors, int k, float* out,
             cudaStream_t stream) {
    const ModePlan& mp = (p.mode[k].path == MTTKRP_PATH_TC && !aligned16(Y)) ? p.simt_alt[k]
                                                                               : p.mode[k];
    const ModeGeom& g = mp.g;
    if (p.ws == nullptr && mp.total > 0)
        return fail(MTTKRP_ERR_WORKSPACE, "no workspace attached (mode %d needs %zu bytes)", k,
                    mp.total);
    if (p.ws_bytes < p.mode[k].total)
        return fail(MTTKRP_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes mode %d needs",
                    p.ws_bytes, p.mode[k].total, k);
    for (int n = 0; n < p.d; ++n)
        if (n != k && factors[n] == nullptr)
            return fail(MTTKRP_ERR_INVALID, "factor %d is NULL", n);
    if (((reinterpret_cast<uintptr_t>(Y) | reinterpret_cast<uintptr_t>(out)) & 3) != 0)
        return fail(MTTKRP_ERR_INVALID, "Y and out must be 4-byte aligned");

    char* ws = static_cast<char*>(p.ws);
    float* partials = reinterpret_cast<float*>(ws + mp.off_partials);
    float* gtab = reinterpret_cast<float*>(ws + mp.off_gtab);
    int64_t* basetab = reinterpret_cast<int64_t*>(ws + mp.off_base);
    cudaError_t err;
    const bool fp16 = mp.path == MTTKRP_PATH_TC && (mp.tc_img || mp.tc_h2);

    // 0. fp16 split: slab maxima of Y and the fp16 images (once per call)
    if (fp16) {
        int nlaunch = 0;
        const int rc = tc_prepare(p, mp, Y, ws, stream, &nlaunch, g_errmsg, sizeof(g_errmsg));
        p.launches += nlaunch;
        if (rc != MTTKRP_OK) return rc;
    }
    // 1. G table and base offsets of the pre indices (fp16 split with per-slab
    //    scales: rows scaled by s_global / s_slab, mode 0 being the first pre mode)
    const bool g_scaled = fp16 && p.slab_on && k != 0;
    auto build_g = [&](const uint32_t* enable) -> int {
        ProdTableArgs a;
        memset(&a, 0, sizeof(a));
        a.nm = g.npm;
        for (int t = 0; t < g.npm; ++t) {
            a.dim[t] = p.dims[g.pm[t]];
            a.ystride[t] = p.strides[g.pm[t]];
            a.fac[t] = factors[g.pm[t]];
        }
        a.rows = g.npre;
        a.R = g.R;
        a.tab = gtab;
        a.base = basetab;
        if (g_scaled) {
            a.slab_bits = reinterpret_cast<const uint32_t*>(ws + p.off_slab);
            a.gmax_bits = reinterpret_cast<const uint32_t*>(ws);
            a.slab_div = g.npre / p.nslab;
        }
        a.enable = enable;
        cudaError_t e = launch_prod_table(a, stream);
        if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "table launch: %s", cudaGetErrorString(e));
        ++p.launches;
        return MTTKRP_OK;
    };
    {
        const int rc = build_g(nullptr);
        if (rc != MTTKRP_OK) return rc;
    }
    float* dst = mp.splits > 1 ? partials : out;
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    if (p.timing) {
        if ((err = timing_pair(p, k, &ev0, &ev1)) != cudaSuccess)
            return fail(MTTKRP_ERR_CUDA, "timing events: %s", cudaGetErrorString(err));
    }

    if (mp.path == MTTKRP_PATH_TC && mp.explicit_krp) {
        // explicit Khatri-Rao product: the table of the group's factors but the
        // last one (the B-image kernel multiplies in the last factor)
        ProdTableArgs a;
        memset(&a, 0, sizeof(a));
        a.nm = g.ngroup - 1;
        for (int t = 0; t + 1 < g.ngroup; ++t) {
            a.dim[t] = p.dims[g.group[t]];
            a.ystride[t] = p.strides[g.group[t]];
            a.fac[t] = factors[g.group[t]];
        }
        a.rows = g.J / p.dims[g.group[g.ngroup - 1]];
        a.R = g.R;
        a.tab = reinterpret_cast<float*>(ws + mp.off_t1);
        if ((err = launch_prod_table(a, stream)) != cudaSuccess)
            return fail(MTTKRP_ERR_CUDA, "table launch: %s", cudaGetErrorString(err));
        ++p.launches;
    }
    if (mp.path == MTTKRP_PATH_TC) {
        int nlaunch = 0;
        if (ev0) cudaEventRecord(ev0, stream);
        int rc = tc_run(p, mp, Y, factors, gtab, basetab, ws + mp.off_binner, dst, stream, &nlaunch,
                        ev0 ? &ev0 : nullptr, g_errmsg, sizeof(g_errmsg));
        p.launches += nlaunch;
        if (rc != MTTKRP_OK) {
            p.fuse_pending = 0;
            return rc;
        }
        if (ev1) {
            cudaEventRecord(ev1, stream);
            ++p.ev_n[k];
        }
        if (p.fuse_pending) {
            // the main kernel converted Y with sampled scales and wrote the
            // images; if a value left the fp16 range, the exact maxima, images,
            // this mode's G table (when it carries slab scales) and its result
            // follow (launches that otherwise return at once)
            rc = tc_redo_images(p, mp, Y, ws, stream, &nlaunch, g_errmsg, sizeof(g_errmsg));
            p.launches += nlaunch;
            if (rc == MTTKRP_OK && g_scaled) rc = build_g(tc_redo_flag(p, ws));
            if (rc == MTTKRP_OK) {
                rc = tc_redo_main(p, mp, Y, factors, gtab, basetab, ws + mp.off_binner, dst, stream, &nlaunch,
                                  g_errmsg, sizeof(g_errmsg));
                p.launches += nlaunch;
            }
            p.fuse_pending = 0;
            if (rc != MTTKRP_OK) return rc;
        }
    } else {
        // 2. Binner (only for an inner group of several modes; else the factor itself)
        const float* binner;
        if (g.ngroup > 1) {
            float* bt = reinterpret_cast<float*>(ws + mp.off_binner);
            ProdTableArgs a;
            memset(&a, 0, sizeof(a));
            a.nm = g.ngroup;
            for (int t = 0; t < g.ngroup; ++t) {
                a.dim[t] = p.dims[g.group[t]];
                a.ystride[t] = p.strides[g.group[t]];
                a.fac[t] = factors[g.group[t]];
            }
            a.rows = g.J;
            a.R = g.R;
            a.tab = bt;
            a.base = nullptr;
            if ((err = launch_prod_table(a, stream)) != cudaSuccess)
                return fail(MTTKRP_ERR_CUDA, "table launch: %s", cudaGetErrorString(err));
            ++p.launches;
            binner = bt;
        } else {
            binner = factors[g.group[0]];
        }
        // 3. main kernel
        SimtArgs a;
        a.Y = Y;
        a.binner = binner;
        a.gtab = gtab;
        a.base = basetab;
        a.dst = dst;
        a.dst_split_stride = g.I * g.R;
        a.I = g.I;
        a.R = g.R;
        a.J = g.J;
        a.Jq = g.Jq;
        a.IQ = g.IQ;
        a.s_k = g.s_k;
        a.npre = g.npre;
        a.pre_per_split = mp.pre_per_split;
        bool strides4 = true;
        for (int t = 0; t < g.npm; ++t) strides4 = strides4 && (p.strides[g.pm[t]] % 4 == 0);
        if (g.J > g.Jq) strides4 = strides4 && (g.IQ % 4 == 0);
        int amode = kLoadScalar;
        if (aligned16(Y) && strides4) {
            if (g.s_k != 1 && g.s_k % 4 == 0 && g.Jq % 4 == 0) amode = kLoadVecJ;
            else if (g.s_k == 1 && g.I % 4 == 0) amode = kLoadVecI;
        }
        const bool bvec = (g.R % 4 == 0) && aligned16(binner);
        if (ev0) cudaEventRecord(ev0, stream);
        if ((err = launch_simt(mp.bm, mp.bn, amode, bvec, a, mp.splits, stream)) != cudaSuccess)
            return fail(MTTKRP_ERR_CUDA, "SIMT kernel launch: %s", cudaGetErrorString(err));
        ++p.launches;
        if (ev1) {
            cudaEventRecord(ev1, stream);
            ++p.ev_n[k];
        }
    }
    // 4. fixed-order reduction of the split partials
    if (mp.splits > 1) {
        if ((err = launch_reduce_splits(partials, mp.splits, g.I * g.R, out, stream)) != cudaSuccess)
            return fail(MTTKRP_ERR_CUDA, "reduce launch: %s", cudaGetErrorString(err));
        ++p.launches;
    }
    return MTTKRP_OK;
}

Plan* as_plan(mttkrp_plan_t h) { return reinterpret_cast<Plan*>(h); }

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" {

int mttkrp_plan(int d, const int64_t* dims, int64_t R, mttkrp_plan_t* out) {
    g_errmsg[0] = 0;
    if (out == nullptr) return fail(MTTKRP_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (d < 2 || d > kMaxD) return fail(MTTKRP_ERR_INVALID, "order d=%d outside [2, %d]", d, kMaxD);
    if (dims == nullptr) return fail(MTTKRP_ERR_INVALID, "dims is NULL");
    if (R < 1 || R > kMaxR) return fail(MTTKRP_ERR_INVALID, "rank R=%lld outside [1, %lld]", (long long)R, (long long)kMaxR);
    int64_t numel = 1;
    for (int n = 0; n < d; ++n) {
        if (dims[n] < 1) return fail(MTTKRP_ERR_INVALID, "dims[%d]=%lld < 1", n, (long long)dims[n]);
        if (dims[n] > kMaxNumel || numel > kMaxNumel / dims[n])
            return fail(MTTKRP_ERR_INVALID, "tensor has more than 2^40 elements");
        numel *= dims[n];
    }
    Plan* p = new (std::nothrow) Plan;
    if (p == nullptr) return fail(MTTKRP_ERR_HOST_ALLOC, "plan allocation failed");
    memset(p, 0, sizeof(*p));
    p->d = d;
    p->R = R;
    for (int n = 0; n < d; ++n) p->dims[n] = dims[n];
    p->strides[d - 1] = 1;
    for (int n = d - 2; n >= 0; --n) p->strides[n] = p->strides[n + 1] * p->dims[n + 1];
    p->forced_path = MTTKRP_PATH_AUTO;
    for (int k = 0; k < d; ++k) {
        int rc = plan_mode(*p, k, MTTKRP_PATH_AUTO);
        if (rc != MTTKRP_OK) {
            delete p;
            return fail(rc, "planning mode %d failed", k);
        }
    }
    place_plan_regions(*p);
    *out = reinterpret_cast<mttkrp_plan_t>(p);
    return MTTKRP_OK;
}

int mttkrp_plan_set_path(mttkrp_plan_t h, int path) {
    Plan* p = as_plan(h);
    if (p == nullptr) return fail(MTTKRP_ERR_INVALID, "plan is NULL");
    if (path != MTTKRP_PATH_AUTO && path != MTTKRP_PATH_SIMT && path != MTTKRP_PATH_TC &&
        path != MTTKRP_PATH_TC_TF32 && path != MTTKRP_PATH_TC_EXPLICIT_KRP)
        return fail(MTTKRP_ERR_INVALID, "unknown path %d", path);
    ModePlan saved[kMaxD];
    memcpy(saved, p->mode, sizeof(saved));
    for (int k = 0; k < p->d; ++k) {
        int rc = plan_mode(*p, k, path);
        if (rc != MTTKRP_OK) {
            memcpy(p->mode, saved, sizeof(saved));
            return fail(rc, "mode %d cannot run on path %d", k, path);
        }
    }
    place_plan_regions(*p);
    p->forced_path = path;
    return MTTKRP_OK;
}

size_t mttkrp_workspace_bytes(mttkrp_plan_t h, int mode) {
    Plan* p = as_plan(h);
    if (p == nullptr || mode < -1 || mode >= p->d) return 0;
    if (mode >= 0) return p->mode[mode].total;
    size_t m = 0;
    for (int k = 0; k < p->d; ++k)
        if (p->mode[k].total > m) m = p->mode[k].total;
    return m;
}

int mttkrp_set_workspace(mttkrp_plan_t h, void* dptr, size_t bytes) {
    Plan* p = as_plan(h);
    if (p == nullptr) return fail(MTTKRP_ERR_INVALID, "plan is NULL");
    if (dptr != nullptr && (reinterpret_cast<uintptr_t>(dptr) & 255) != 0)
        return fail(MTTKRP_ERR_INVALID, "workspace must be 256-byte aligned");
    p->ws = dptr;
    p->ws_bytes = dptr ? bytes : 0;
    p->sweep_left_images = 0;   // a new workspace holds none of the earlier results
    return MTTKRP_OK;
}

int mttkrp(mttkrp_plan_t h, const float* Y, const float* const* factors, int mode, float* out,
           void* stream) {
    g_errmsg[0] = 0;
    Plan* p = as_plan(h);
    if (p == nullptr) return fail(MTTKRP_ERR_INVALID, "plan is NULL");
    if (mode < 0 || mode >= p->d) return fail(MTTKRP_ERR_INVALID, "mode %d outside [0, %d)", mode, p->d);
    if (Y == nullptr || factors == nullptr || out == nullptr)
        return fail(MTTKRP_ERR_INVALID, "NULL tensor, factor array or output");
    p->ymax_ready = 0;
    p->img_ready = 0;
    p->fuse_pending = 0;
    p->sweep_left_images = 0;
    return run_mode(*p, Y, factors, mode, out, static_cast<cudaStream_t>(stream));
}

int mttkrp_all_modes(mttkrp_plan_t h, const float* Y, const float* const* factors,
                     float* const* outs, void* stream) {
    g_errmsg[0] = 0;
    Plan* p = as_plan(h);
    if (p == nullptr) return fail(MTTKRP_ERR_INVALID, "plan is NULL");
    if (Y == nullptr || factors == nullptr || outs == nullptr)
        return fail(MTTKRP_ERR_INVALID, "NULL tensor, factor array or output array");
    for (int k = 0; k < p->d; ++k) {
        if (factors[k] == nullptr) return fail(MTTKRP_ERR_INVALID, "factor %d is NULL", k);
        if (outs[k] == nullptr) return fail(MTTKRP_ERR_INVALID, "output %d is NULL", k);
    }
    p->ymax_ready = 0;   // one max |Y| pass serves every mode of this call
    p->img_ready = 0;    // and one pass writing the fp16 images of Y
    p->fuse_pending = 0;
    p->sweep_left_images = 0;
    // the mode that converts Y and writes the images (if any) first, then the
    // others in order (each mode's result does not depend on the order)
    const int first = p->fuse_mode;
    for (int t = -1; t < p->d; ++t) {
        const int k = t < 0 ? first : t;
        if (k < 0 || (t >= 0 && k == first)) continue;
        int rc = run_mode(*p, Y, factors, k, outs[k], static_cast<cudaStream_t>(stream));
        if (rc != MTTKRP_OK) return rc;
    }
    return MTTKRP_OK;
}

// CP-ALS scratch: Gram matrices of every mode, V (reused for the Hadamard
// product of all Grams), the fp64 solve of the current mode, its fp32 MTTKRP,
// the ||Y||^2 and fit partials, the Cholesky status word, and for the
// mixed-precision solve (R <= cpals_mixed_max_rank()) V's two fp32 words, the
// fp32 factor and the fp32 first solution and residual.
namespace {
struct CpAlsLayout {
    size_t grams, v, dinv, x, m, gpart, part, npart, info, vhi, vlo, l32, dinv32, dblk, x0, res, total;
};
CpAlsLayout cp_als_layout(const Plan& p) {
    int64_t imax = 0;
    for (int n = 0; n < p.d; ++n) imax = p.dims[n] > imax ? p.dims[n] : imax;
    const size_t R = (size_t)p.R;
    CpAlsLayout l;
    size_t off = 0;
    l.grams = off;
    off = align256(off + (size_t)p.d * R * R * sizeof(double));
    l.v = off;
    off = align256(off + R * R * sizeof(double));
    l.dinv = off;
    off = align256(off + R * sizeof(double));
    l.x = off;
    off = align256(off + (size_t)imax * R * sizeof(double));
    l.m = off;
    off = align256(off + (size_t)imax * R * sizeof(float));
    int slabs = 1;
    for (int n = 0; n < p.d; ++n) {
        const int sn = cpals_gram_slabs(p.dims[n], (int)p.R);
        slabs = sn > slabs ? sn : slabs;
    }
    l.gpart = off;
    off = align256(off + (slabs > 1 ? (size_t)slabs * R * R * sizeof(double) : 0));
    l.part = off;
    off = align256(off + cpals_sumsq_scratch_bytes());
    l.npart = off;
    off = align256(off + cpals_normalize_scratch_bytes((int)p.R));
    l.info = off;
    off = align256(off + sizeof(int));
    const bool mixed = p.R <= cpals_mixed_max_rank();
    l.vhi = off;
    off = align256(off + (mixed ? R * R * sizeof(float) : 0));
    l.vlo = off;
    off = align256(off + (mixed ? R * R * sizeof(float) : 0));
    l.l32 = off;
    off = align256(off + (mixed ? R * R * sizeof(float) : 0));
    l.dinv32 = off;
    off = align256(off + (mixed ? R * sizeof(float) : 0));
    l.dblk = off;
    off = align256(off + (mixed ? cpals_mixed_block_bytes((int)p.R) : 0));
    l.x0 = off;
    off = align256(off + (mixed ? (size_t)imax * R * sizeof(float) : 0));
    l.res = off;
    off = align256(off + (mixed ? (size_t)imax * R * sizeof(float) : 0));
    l.total = off;
    return l;
}
}  // namespace

int mttkrp_apply_rotations(int d, const int64_t* dims, float* Y, int mode, const int32_t* pairs, const float* c,
                           const float* s, int group_size, void* stream) {
    g_errmsg[0] = 0;
    if (d < 2 || d > kMaxD) return fail(MTTKRP_ERR_INVALID, "order d=%d outside [2, %d]", d, kMaxD);
    if (dims == nullptr || Y == nullptr) return fail(MTTKRP_ERR_INVALID, "NULL dims or tensor");
    if (mode < 0 || mode >= d) return fail(MTTKRP_ERR_INVALID, "mode %d outside [0, %d)", mode, d);
    int64_t P = 1, Q = 1, numel = 1;
    for (int n = 0; n < d; ++n) {
        if (dims[n] < 1) return fail(MTTKRP_ERR_INVALID, "dims[%d]=%lld < 1", n, (long long)dims[n]);
        if (dims[n] > kMaxNumel || numel > kMaxNumel / dims[n])
            return fail(MTTKRP_ERR_INVALID, "tensor has more than 2^40 elements");
        numel *= dims[n];
        if (n < mode) P *= dims[n];
        if (n > mode) Q *= dims[n];
    }
    const int64_t N = dims[mode];
    if (N > INT32_MAX) return fail(MTTKRP_ERR_INVALID, "mode size %lld too large", (long long)N);
    if (group_size < 0 || 2 * (int64_t)group_size > N)
        return fail(MTTKRP_ERR_INVALID, "group of %d disjoint pairs does not fit mode size %lld", group_size,
                    (long long)N);
    if (group_size > 0 && (pairs == nullptr || c == nullptr || s == nullptr))
        return fail(MTTKRP_ERR_INVALID, "NULL pairs, cosines or sines");
    if ((reinterpret_cast<uintptr_t>(Y) & 3) != 0) return fail(MTTKRP_ERR_INVALID, "Y must be 4-byte aligned");
    cudaError_t e = launch_rotations(Y, P, (int)N, Q, pairs, c, s, group_size, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "rotation launch: %s", cudaGetErrorString(e));
    return MTTKRP_OK;
}

}  // extern "C"

namespace mk {
namespace {
// Argument checks of the mode-n product; P, N, Q of X viewed [P, N, Q].
int ttm_check(int d, const int64_t* dims, const float* X, int mode, const float* M, int64_t J, const float* T,
              int64_t* Pout, int64_t* Nout, int64_t* Qout) {
    if (d < 1 || d > kMaxD) return fail(MTTKRP_ERR_INVALID, "order d=%d outside [1, %d]", d, kMaxD);
    if (dims == nullptr || X == nullptr || M == nullptr || T == nullptr)
        return fail(MTTKRP_ERR_INVALID, "NULL dims, tensor, matrix or result");
    if (mode < 0 || mode >= d) return fail(MTTKRP_ERR_INVALID, "mode %d outside [0, %d)", mode, d);
    if (J < 1 || J > ((int64_t)1 << 24))
        return fail(MTTKRP_ERR_INVALID, "J=%lld outside [1, 2^24]", (long long)J);
    int64_t P = 1, Q = 1, numel = 1;
    for (int n = 0; n < d; ++n) {
        if (dims[n] < 1) return fail(MTTKRP_ERR_INVALID, "dims[%d]=%lld < 1", n, (long long)dims[n]);
        if (dims[n] > kMaxNumel || numel > kMaxNumel / dims[n])
            return fail(MTTKRP_ERR_INVALID, "tensor has more than 2^40 elements");
        numel *= dims[n];
        if (n < mode) P *= dims[n];
        if (n > mode) Q *= dims[n];
    }
    const int64_t N = dims[mode];
    if (P * Q > kMaxNumel / J) return fail(MTTKRP_ERR_INVALID, "result has more than 2^40 elements");
    if (ttm_tiles(P, Q, J) > INT32_MAX) return fail(MTTKRP_ERR_INVALID, "too many result tiles");
    if (((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(M) | reinterpret_cast<uintptr_t>(T)) & 3) != 0)
        return fail(MTTKRP_ERR_INVALID, "X, M and T must be 4-byte aligned");
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(X), x1 = x0 + (uintptr_t)numel * 4;
    const uintptr_t t0 = reinterpret_cast<uintptr_t>(T), t1 = t0 + (uintptr_t)(P * J * Q) * 4;
    const uintptr_t m0 = reinterpret_cast<uintptr_t>(M), m1 = m0 + (uintptr_t)(J * N) * 4;
    if ((t0 < x1 && x0 < t1) || (t0 < m1 && m0 < t1))
        return fail(MTTKRP_ERR_INVALID, "the result overlaps X or M");
    *Pout = P;
    *Nout = N;
    *Qout = Q;
    return MTTKRP_OK;
}
}  // namespace
}  // namespace mk

extern "C" {

int mttkrp_ttm(int d, const int64_t* dims, const float* X, int mode, const float* M, int64_t J, float* T,
               void* stream) {
    g_errmsg[0] = 0;
    int64_t P, N, Q;
    const int rc = ttm_check(d, dims, X, mode, M, J, T, &P, &N, &Q);
    if (rc != MTTKRP_OK) return rc;
    cudaError_t e = launch_ttm(X, M, T, P, N, Q, J, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "mode-n product launch: %s", cudaGetErrorString(e));
    return MTTKRP_OK;
}

size_t mttkrp_ttm_workspace_bytes(int d, const int64_t* dims, int mode, int64_t J) {
    if (d < 1 || d > kMaxD || dims == nullptr || mode < 0 || mode >= d || J < 1) return 0;
    int64_t P = 1, Q = 1, numel = 1;
    for (int n = 0; n < d; ++n) {
        if (dims[n] < 1 || dims[n] > kMaxNumel || numel > kMaxNumel / dims[n]) return 0;
        numel *= dims[n];
        if (n < mode) P *= dims[n];
        if (n > mode) Q *= dims[n];
    }
    return tc_ttm_workspace_bytes(P, dims[mode], Q, J);
}

int mttkrp_ttm_ws(int d, const int64_t* dims, const float* X, int mode, const float* M, int64_t J, float* T,
                  void* workspace, size_t workspace_bytes, void* stream) {
    g_errmsg[0] = 0;
    int64_t P, N, Q;
    const int rc = ttm_check(d, dims, X, mode, M, J, T, &P, &N, &Q);
    if (rc != MTTKRP_OK) return rc;
    const size_t need = tc_ttm_workspace_bytes(P, N, Q, J);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (need > 0 && workspace != nullptr && workspace_bytes >= need &&
        (reinterpret_cast<uintptr_t>(X) & 15) == 0 && (reinterpret_cast<uintptr_t>(workspace) & 255) == 0)
        return tc_ttm_run(X, M, T, P, N, Q, J, workspace, s, g_errmsg, sizeof(g_errmsg));
    if (need > 0 && workspace != nullptr && workspace_bytes < need)
        return fail(MTTKRP_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes,
                    need);
    cudaError_t e = launch_ttm(X, M, T, P, N, Q, J, s);
    if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "mode-n product launch: %s", cudaGetErrorString(e));
    return MTTKRP_OK;
}

size_t mttkrp_ttm_multi_workspace_bytes(int d, const int64_t* dims, int nmodes, const int* modes,
                                        const int64_t* Js) {
    if (nmodes < 1 || nmodes > 64 || modes == nullptr || Js == nullptr) return 0;
    size_t need = 0;
    for (int t = 0; t < nmodes; ++t) {
        const size_t b = mttkrp_ttm_workspace_bytes(d, dims, modes[t], Js[t]);
        if (b > need) need = b;   // images at the same offsets for every product of one X
    }
    return need;
}

int mttkrp_ttm_multi(int d, const int64_t* dims, const float* X, int nmodes, const int* modes,
                     const float* const* Ms, const int64_t* Js, float* const* Ts, void* workspace,
                     size_t workspace_bytes, void* stream) {
    g_errmsg[0] = 0;
    if (nmodes < 1 || nmodes > 64) return fail(MTTKRP_ERR_INVALID, "nmodes=%d outside [1, 64]", nmodes);
    if (modes == nullptr || Ms == nullptr || Js == nullptr || Ts == nullptr)
        return fail(MTTKRP_ERR_INVALID, "NULL modes, matrices, row counts or results");
    int64_t P[64], N[64], Q[64];
    size_t need[64];
    for (int t = 0; t < nmodes; ++t) {
        const int rc = ttm_check(d, dims, X, modes[t], Ms[t], Js[t], Ts[t], &P[t], &N[t], &Q[t]);
        if (rc != MTTKRP_OK) return rc;
        need[t] = tc_ttm_workspace_bytes(P[t], N[t], Q[t], Js[t]);
    }
    // a later product must not overwrite an earlier one's result or matrix
    for (int t = 0; t < nmodes; ++t) {
        const uintptr_t t0 = reinterpret_cast<uintptr_t>(Ts[t]), t1 = t0 + (uintptr_t)(P[t] * Js[t] * Q[t]) * 4;
        for (int u = 0; u < nmodes; ++u) {
            if (u == t) continue;
            const uintptr_t u0 = reinterpret_cast<uintptr_t>(Ts[u]), u1 = u0 + (uintptr_t)(P[u] * Js[u] * Q[u]) * 4;
            const uintptr_t m0 = reinterpret_cast<uintptr_t>(Ms[u]), m1 = m0 + (uintptr_t)(Js[u] * N[u]) * 4;
            if ((t0 < u1 && u0 < t1) || (t0 < m1 && m0 < t1))
                return fail(MTTKRP_ERR_INVALID, "result %d overlaps result or matrix %d", t, u);
        }
    }
    size_t need_all = 0;
    for (int t = 0; t < nmodes; ++t) need_all = need[t] > need_all ? need[t] : need_all;
    if (workspace != nullptr && need_all > 0 && workspace_bytes < need_all)
        return fail(MTTKRP_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes,
                    need_all);
    const bool tc_ok = workspace != nullptr && (reinterpret_cast<uintptr_t>(X) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(workspace) & 255) == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool images = false;
    for (int t = 0; t < nmodes; ++t) {
        if (tc_ok && need[t] > 0) {
            if (!images) {
                const int rc = tc_ttm_images(X, P[t] * N[t] * Q[t], workspace, s, g_errmsg, sizeof(g_errmsg));
                if (rc != MTTKRP_OK) return rc;
                images = true;
            }
            const int rc = tc_ttm_product(Ms[t], Ts[t], P[t], N[t], Q[t], Js[t], workspace, s, g_errmsg,
                                          sizeof(g_errmsg));
            if (rc != MTTKRP_OK) return rc;
        } else {
            cudaError_t e = launch_ttm(X, Ms[t], Ts[t], P[t], N[t], Q[t], Js[t], s);
            if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "mode-n product launch: %s", cudaGetErrorString(e));
        }
    }
    return MTTKRP_OK;
}

size_t mttkrp_cp_als_scratch_bytes(mttkrp_plan_t h) {
    Plan* p = as_plan(h);
    return p == nullptr ? 0 : cp_als_layout(*p).total;
}

int mttkrp_cp_als_sweep(mttkrp_plan_t h, const float* Y, float* const* factors, float* lambda,
                        double* norm_y2, int have_norm, double* fit, void* scratch, size_t scratch_bytes,
                        void* stream) {
    g_errmsg[0] = 0;
    Plan* p = as_plan(h);
    if (p == nullptr) return fail(MTTKRP_ERR_INVALID, "plan is NULL");
    if (Y == nullptr || factors == nullptr || lambda == nullptr || norm_y2 == nullptr || fit == nullptr ||
        scratch == nullptr)
        return fail(MTTKRP_ERR_INVALID, "NULL tensor, factor array, lambda, norm, fit or scratch");
    for (int n = 0; n < p->d; ++n)
        if (factors[n] == nullptr) return fail(MTTKRP_ERR_INVALID, "factor %d is NULL", n);
    if ((reinterpret_cast<uintptr_t>(scratch) & 255) != 0)
        return fail(MTTKRP_ERR_INVALID, "scratch must be 256-byte aligned");
    if (p->R > 65535) return fail(MTTKRP_ERR_UNSUPPORTED, "CP-ALS rank %lld above 65535", (long long)p->R);
    const CpAlsLayout l = cp_als_layout(*p);
    if (scratch_bytes < l.total)
        return fail(MTTKRP_ERR_WORKSPACE, "CP-ALS scratch of %zu bytes is smaller than the %zu bytes needed",
                    scratch_bytes, l.total);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(scratch);
    double* G = reinterpret_cast<double*>(base + l.grams);
    double* V = reinterpret_cast<double*>(base + l.v);
    double* dinv = reinterpret_cast<double*>(base + l.dinv);
    double* X = reinterpret_cast<double*>(base + l.x);
    float* M = reinterpret_cast<float*>(base + l.m);
    double* part = reinterpret_cast<double*>(base + l.part);
    double* gpart = reinterpret_cast<double*>(base + l.gpart);
    int* info = reinterpret_cast<int*>(base + l.info);
    const int d = p->d;
    const int R = (int)p->R;
    const int64_t RR = (int64_t)R * R;
    const bool mixed = R <= cpals_mixed_max_rank();
    int64_t numel = 1;
    for (int n = 0; n < d; ++n) numel *= p->dims[n];
    cudaError_t e = cudaMemsetAsync(info, 0, sizeof(int), s);
    if (e == cudaSuccess && !have_norm) {
        e = cpals_sum_squares(Y, numel, part, norm_y2, s);
        p->launches += 2;
    }
    // the Gram matrix of every factor; a continuing sweep on the same scratch and
    // factors finds them where the previous sweep left them (each computed right
    // after its factor's last update)
    bool grams_ready = have_norm && p->sweep_left_images && p->sweep_scratch == scratch;
    for (int n = 0; n < d; ++n) grams_ready = grams_ready && p->sweep_factors[n] == factors[n];
    for (int n = 0; n < d && e == cudaSuccess && !grams_ready; ++n) {
        e = cpals_gram(factors[n], p->dims[n], R, G + n * RR, gpart, s);
        p->launches += cpals_gram_slabs(p->dims[n], R) > 1 ? 2 : 1;
    }
    if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "CP-ALS setup: %s", cudaGetErrorString(e));
    // one max |Y| pass and one image pass serve every mode of the sweep; a
    // continuing sweep (have_norm: the same Y, no other call on the plan since
    // the previous sweep) reuses the previous sweep's
    const int reuse = have_norm && p->sweep_left_images;
    p->ymax_ready = reuse;
    p->img_ready = reuse;
    p->fuse_pending = 0;
    p->sweep_left_images = 0;
    for (int n = 0; n < d; ++n) {
        float* vhi = mixed ? reinterpret_cast<float*>(base + l.vhi) : nullptr;
        float* vlo = mixed ? reinterpret_cast<float*>(base + l.vlo) : nullptr;
        if ((e = cpals_hadamard(G, d, n, R, V, vhi, vlo, s)) != cudaSuccess)
            return fail(MTTKRP_ERR_CUDA, "CP-ALS Hadamard: %s", cudaGetErrorString(e));
        ++p->launches;
        int rc = run_mode(*p, Y, factors, n, M, s);
        if (rc != MTTKRP_OK) return rc;
        if (mixed) {
            e = cpals_solve_mixed(V, R, M, p->dims[n], X, reinterpret_cast<float*>(base + l.vhi),
                                  reinterpret_cast<float*>(base + l.vlo), reinterpret_cast<float*>(base + l.l32),
                                  reinterpret_cast<float*>(base + l.dinv32), reinterpret_cast<float*>(base + l.dblk),
                                  reinterpret_cast<float*>(base + l.x0),
                                  reinterpret_cast<float*>(base + l.res), info, s);
            p->launches += cpals_mixed_launches(R);
        } else {
            if ((e = cpals_cholesky(V, R, info, dinv, s)) == cudaSuccess)
                e = cpals_solve(V, dinv, R, M, p->dims[n], X, s);
            p->launches += 2 + cpals_cholesky_launches(R);
        }
        if (e == cudaSuccess &&
            (e = cpals_normalize(X, p->dims[n], R, factors[n], lambda, reinterpret_cast<double*>(base + l.npart), s)) ==
                cudaSuccess)
            e = cpals_gram(factors[n], p->dims[n], R, G + n * RR, gpart, s);
        if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "CP-ALS update of mode %d: %s", n, cudaGetErrorString(e));
        p->launches += cpals_normalize_launches() + 1 + (cpals_gram_slabs(p->dims[n], R) > 1 ? 1 : 0);
    }
    if ((e = cpals_hadamard(G, d, -1, R, V, nullptr, nullptr, s)) == cudaSuccess)
        e = cpals_fit(V, lambda, M, factors[d - 1], p->dims[d - 1], R, norm_y2, info, fit, part, s);
    if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "CP-ALS fit: %s", cudaGetErrorString(e));
    p->launches += 3;
    p->sweep_left_images = 1;
    p->sweep_scratch = scratch;
    for (int n = 0; n < d; ++n) p->sweep_factors[n] = factors[n];
    return MTTKRP_OK;
}

int mttkrp_plan_mode_path(mttkrp_plan_t h, int mode) {
    Plan* p = as_plan(h);
    if (p == nullptr || mode < 0 || mode >= p->d) return -1;
    return p->mode[mode].path;
}

int mttkrp_plan_describe(mttkrp_plan_t h, int mode, char* buf, size_t len) {
    Plan* p = as_plan(h);
    if (p == nullptr || mode < 0 || mode >= p->d) return -1;
    const ModePlan& mp = p->mode[mode];
    const ModeGeom& g = mp.g;
    char groups[64] = "", pres[64] = "";
    for (int t = 0; t < g.ngroup; ++t)
        snprintf(groups + strlen(groups), sizeof(groups) - strlen(groups), "%s%d", t ? "," : "", g.group[t]);
    for (int t = 0; t < g.npm; ++t)
        snprintf(pres + strlen(pres), sizeof(pres) - strlen(pres), "%s%d", t ? "," : "", g.pm[t]);
    // kernel variant: family (simt; img = fp16 images, h2 = fp16 split in tensor
    // memory, tf32 = 3xTF32 with A in shared memory, tf32tm = 3xTF32 with A in
    // tensor memory), then the A layout (nat / t = transposed images, kmaj / inner
    // = raw fp32 tiles), "small" for stacked pre indices, and the tile width
    char kernel[64];
    if (mp.path != MTTKRP_PATH_TC) {
        snprintf(kernel, sizeof(kernel), "simt.bn%d", mp.bn);
    } else {
        const char* fam = mp.tc_img ? "img" : mp.tc_h2 ? "h2" : mp.tc_tmem ? "tf32tm" : "tf32";
        const char* lay = mp.tc_img ? (mp.tc_img_t ? "t" : mp.tc_img_mn ? "mn" : "nat")
                                    : (mp.tc_inner ? "inner" : "kmaj");
        snprintf(kernel, sizeof(kernel), "%s.%s%s.bn%d", fam, lay, mp.tc_small ? ".small" : "", mp.bn);
    }
    // fp32 bytes of the explicit Khatri-Rao product of every mode but this one
    // (what the matrix-based variant forms; the matrix-free one never does)
    int64_t others = 1;
    for (int t = 0; t < p->d; ++t)
        if (t != mode) others *= p->dims[t];
    const double krp_bytes = 4.0 * (double)p->R * (double)others;
    // workspace by purpose: split partial sums; tables (factor products, the B
    // operand images -- for the explicit variant the whole Khatri-Rao product);
    // plan-wide fp16 images of Y and slab maxima (fp16-split modes)
    const bool fp16 = mp.path == MTTKRP_PATH_TC && (mp.tc_img || mp.tc_h2);
    const size_t ws_images = fp16 ? mp.total - p->off_slab : 0;
    char tmp[640];
    int n = snprintf(tmp, sizeof(tmp),
                     "mode=%d path=%s kernel=%s tile=%dx%d inner_group=[%s] J=%lld Jq=%lld pre_modes=[%s] "
                     "npre=%lld splits=%lld pre_per_split=%lld workspace=%zu tc_ksteps=%d tc_inner=%d tc_slots=%d "
                     "tc_tmem_a=%d tc_fp16x2=%d tc_fp16_image=%d krp=%s krp_bytes=%llu "
                     "ws_partials=%zu ws_tables=%zu ws_images=%zu tc_convert=%d",
                     mode, mp.path == MTTKRP_PATH_TC ? "tc" : "simt", kernel, mp.bm, mp.bn, groups,
                     (long long)g.J, (long long)g.Jq, pres, (long long)g.npre,
                     (long long)mp.splits, (long long)mp.pre_per_split, mp.total, mp.tc_ks, mp.tc_inner,
                     mp.tc_small ? mp.tc_ps : 1, mp.tc_tmem, mp.tc_h2 || mp.tc_img,
                     mp.tc_img ? (mp.tc_img_t ? 2 : mp.tc_img_mn ? 3 : 1) : 0,
                     mp.explicit_krp ? "explicit" : "free", (unsigned long long)krp_bytes,
                     mp.off_binner - mp.off_partials, mp.off_end - mp.off_binner, ws_images,
                     mode == p->fuse_mode ? 1 : 0);
    if (buf != nullptr && len > 0) {
        strncpy(buf, tmp, len - 1);
        buf[len - 1] = 0;
    }
    return n;
}

int mttkrp_device_status(uint32_t* word) {
    if (word == nullptr) return fail(MTTKRP_ERR_INVALID, "word is NULL");
    cudaError_t err = tc_read_and_clear_status(word);
    if (err != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "status read: %s", cudaGetErrorString(err));
    return MTTKRP_OK;
}

int mttkrp_plan_set_timing(mttkrp_plan_t h, int enable) {
    Plan* p = as_plan(h);
    if (p == nullptr) return -fail(MTTKRP_ERR_INVALID, "plan is NULL");
    p->timing = enable ? 1 : 0;
    for (int k = 0; k < kMaxD; ++k) p->ev_n[k] = 0;
    return MTTKRP_OK;
}

int mttkrp_plan_kernel_times(mttkrp_plan_t h, int mode, float* ms, int max) {
    Plan* p = as_plan(h);
    if (p == nullptr || mode < 0 || mode >= p->d || (ms == nullptr && max > 0))
        return -fail(MTTKRP_ERR_INVALID, "invalid plan, mode or buffer");
    const int n = p->ev_n[mode];
    for (int i = 0; i < n && i < max; ++i) {
        cudaError_t err = cudaEventSynchronize(p->ev_stop[mode][i]);
        if (err == cudaSuccess) err = cudaEventElapsedTime(&ms[i], p->ev_start[mode][i], p->ev_stop[mode][i]);
        if (err != cudaSuccess) return -fail(MTTKRP_ERR_CUDA, "event timing: %s", cudaGetErrorString(err));
    }
    return n;
}

int64_t mttkrp_plan_launch_count(mttkrp_plan_t h) {
    Plan* p = as_plan(h);
    return p ? p->launches : -1;
}

int mttkrp_test_withhold_signal(int count) { return tc_set_withhold_signal(count); }

void mttkrp_plan_destroy(mttkrp_plan_t h) {
    Plan* p = as_plan(h);
    if (p == nullptr) return;
    free_events(*p);
    delete p;
}

const char* mttkrp_strerror(int code) {
    switch (code) {
        case MTTKRP_OK: return "ok";
        case MTTKRP_ERR_INVALID: return "invalid argument";
        case MTTKRP_ERR_UNSUPPORTED: return "unsupported on the requested path";
        case MTTKRP_ERR_WORKSPACE: return "workspace missing or too small";
        case MTTKRP_ERR_CUDA: return "CUDA error";
        case MTTKRP_ERR_HOST_ALLOC: return "host allocation failed";
        case MTTKRP_ERR_DEVICE: return "device-side error (bounded wait expired)";
        default: return "unknown error code";
    }
}

const char* mttkrp_last_error(void) { return g_errmsg; }

int mttkrp_version(void) { return 100; }

int mttkrp_probe_fma(int blocks, int iters, float* out, void* stream) {
    g_errmsg[0] = 0;
    if (blocks < 1 || blocks > 65535 || iters < 1 || out == nullptr)
        return fail(MTTKRP_ERR_INVALID, "blocks in [1, 65535], iters >= 1 and a non-NULL out are required");
    cudaError_t e = launch_fma_probe(blocks, iters, out, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "FMA probe launch: %s", cudaGetErrorString(e));
    return MTTKRP_OK;
}

int mttkrp_probe_mma(int kind, int blocks, int iters, void* stream) {
    g_errmsg[0] = 0;
    if ((kind != 0 && kind != 1) || blocks < 1 || blocks > 65535 || iters < 1)
        return fail(MTTKRP_ERR_INVALID, "kind 0 (tf32) or 1 (f16), blocks in [1, 65535] and iters >= 1 are required");
    cudaError_t e = tc_launch_mma_probe(kind, blocks, iters, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MTTKRP_ERR_CUDA, "MMA probe launch: %s", cudaGetErrorString(e));
    return MTTKRP_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (mttkrp_noalloc).
//
// Some callers cannot call cudaMalloc: a library embedded in a host program
// whose own allocator reserves and hands out all device memory (a framework's
// caching allocator, an inference server's arena) and forbids foreign
// allocations, or code on a latency-critical path where cudaMalloc/cudaFree,
// which can block until the device is idle, are not acceptable.  For them the
// scratch that the SIMT path needs (split partial sums, factor-product
// tables) lives in one fixed, file-scope device array instead of a
// caller-provided workspace.  The array is part of the library image: every
// GPU that loads the library holds it until the process exits.
// ---------------------------------------------------------------------------

#include <mutex>

namespace mk {

static __device__ __align__(256) unsigned char g_static_scratch[MTTKRP_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  The host-side
// name of the array is only a stand-in, never a device address, so the address
// is looked up once per device (with that device current) and cached.
cudaError_t static_scratch_address(void** out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_static_scratch);
        if (err != cudaSuccess) return err;
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace mk

extern "C" int mttkrp_noalloc(int d, const int64_t* dims, int64_t R, const float* Y,
                              const float* const* factors, int mode, float* out, void* stream) {
    g_errmsg[0] = 0;
    if (d < 2 || d > kMaxD) return fail(MTTKRP_ERR_INVALID, "order d=%d outside [2, %d]", d, kMaxD);
    if (dims == nullptr || Y == nullptr || factors == nullptr || out == nullptr)
        return fail(MTTKRP_ERR_INVALID, "NULL dims, tensor, factor array or output");
    if (R < 1 || R > kMaxR) return fail(MTTKRP_ERR_INVALID, "rank R=%lld outside [1, %lld]", (long long)R, (long long)kMaxR);
    if (mode < 0 || mode >= d) return fail(MTTKRP_ERR_INVALID, "mode %d outside [0, %d)", mode, d);
    int64_t numel = 1;
    for (int n = 0; n < d; ++n) {
        if (dims[n] < 1) return fail(MTTKRP_ERR_INVALID, "dims[%d]=%lld < 1", n, (long long)dims[n]);
        if (dims[n] > kMaxNumel || numel > kMaxNumel / dims[n])
            return fail(MTTKRP_ERR_INVALID, "tensor has more than 2^40 elements");
        numel *= dims[n];
    }
    // the plan lives on the stack: nothing is allocated, on the host or the GPU
    Plan p;
    memset(&p, 0, sizeof(p));
    p.d = d;
    p.R = R;
    for (int n = 0; n < d; ++n) p.dims[n] = dims[n];
    p.strides[d - 1] = 1;
    for (int n = d - 2; n >= 0; --n) p.strides[n] = p.strides[n + 1] * p.dims[n + 1];
    p.forced_path = MTTKRP_PATH_SIMT;
    p.fuse_mode = -1;
    int rc = plan_mode(p, mode, MTTKRP_PATH_SIMT);
    if (rc != MTTKRP_OK) return fail(rc, "mode %d cannot be planned on the SIMT path", mode);
    const size_t need = p.mode[mode].total;
    if (need > (size_t)MTTKRP_NOALLOC_SCRATCH_BYTES)
        return fail(MTTKRP_ERR_WORKSPACE,
                    "mttkrp_noalloc: this problem needs %zu bytes of scratch, more than the "
                    "%zu-byte static scratch; use mttkrp() with a workspace instead",
                    need, (size_t)MTTKRP_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    cudaError_t err = static_scratch_address(&scratch);
    if (err != cudaSuccess)
        return fail(MTTKRP_ERR_CUDA, "static scratch address: %s", cudaGetErrorString(err));
    p.ws = scratch;
    p.ws_bytes = MTTKRP_NOALLOC_SCRATCH_BYTES;
    return run_mode(p, Y, factors, mode, out, static_cast<cudaStream_t>(stream));
}
