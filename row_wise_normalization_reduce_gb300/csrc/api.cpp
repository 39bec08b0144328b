// api.cpp -- the C ABI (include/nrm.h): argument validation, the per-shape
// plan choice and the launches.  Argument checks follow the extension
// boundary of the CUDA fused RMSNorm kernel page (diycv.top, §5: device,
// contiguity, shape and type checks, current stream, launch check) and the
// edge-case list of the LayerNorm walkthrough (lpnh.cn/news/2756757, §7:
// N not a multiple of the vector width, optional gamma/beta, no in-place
// y == x, check the launch).
#include <cuda_runtime_api.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "nrm.h"
#include "nrm_internal.h"

using namespace nrm;

namespace {

// ---------------------------------------------------------------------------
// Device attributes, queried once per device.
// ---------------------------------------------------------------------------
struct DevInfo {
    int sms = 0;
    bool ok = false;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

int device_info(DevInfo *out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NRM_ERR_DEVICE;
    }
    std::call_once(g_dev_once[dev], [dev]() {
        DevInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            d.sms > 0)
            d.ok = true;
        else
            cudaGetLastError();
        g_dev[dev] = d;
    });
    if (!g_dev[dev].ok) return NRM_ERR_DEVICE;
    *out = g_dev[dev];
    return NRM_OK;
}

std::atomic<int> g_force_kind{0}, g_force_threads{0}, g_force_packs{0}, g_force_stages{0},
    g_force_groups{0};
std::atomic<unsigned> g_wait_limit{1u << 20};
std::atomic<int> g_pointer_checks{0};
// 0 = no grouping: one group of all channels (measured fastest at both
// [32, 64, 56, 56] and [64, 64, 112, 112]; smaller groups only added the
// statistics-to-normalize serialization once per group)
std::atomic<size_t> g_bn_group_bytes{0};
thread_local int t_last_kind = 0, t_last_threads = 0, t_last_packs = 0, t_last_stages = 0,
                 t_last_groups = 0;

size_t elem_size(int dtype) { return dtype == NRM_F32 ? 4 : 2; }
bool dtype_ok(int dtype) { return dtype == NRM_F32 || dtype == NRM_F16 || dtype == NRM_BF16; }

// [p, p + bytes) as integers, for overlap tests.
struct Span {
    uintptr_t lo = 0, hi = 0;
    bool live() const { return hi > lo; }
};
Span span(const void *p, size_t bytes) {
    Span s;
    if (p && bytes) {
        s.lo = reinterpret_cast<uintptr_t>(p);
        s.hi = s.lo + bytes;
    }
    return s;
}
bool overlap(const Span &a, const Span &b) {
    return a.live() && b.live() && a.lo < b.hi && b.lo < a.hi;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_pointer(const void *p) {
    if (!p) return NRM_OK;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return NRM_ERR_POINTER;
    }
    int dev = -1;
    cudaGetDevice(&dev);
    if (attr.type == cudaMemoryTypeManaged) return NRM_OK;
    if (attr.type != cudaMemoryTypeDevice || attr.device != dev) return NRM_ERR_POINTER;
    return NRM_OK;
}

int check_pointers(std::initializer_list<const void *> ps) {
    if (!g_pointer_checks.load(std::memory_order_relaxed)) return NRM_OK;
    for (const void *p : ps) {
        int st = check_pointer(p);
        if (st != NRM_OK) return st;
    }
    return NRM_OK;
}

bool eps_ok(float eps) { return std::isfinite(eps) && eps >= 0.f; }

// BatchNorm plan from the forced row plan (a test and measurement hook):
// GENERIC -> scalar two kernels, TMA -> cluster per channel, CTA -> streaming.
int bn_plan_from_forced() {
    switch (g_force_kind.load(std::memory_order_relaxed)) {
    case PLAN_GENERIC: return BN_PLAN_SCALAR;
    case PLAN_TMA: return BN_PLAN_CLUSTER;
    case PLAN_CTA: return BN_PLAN_STREAM;
    case PLAN_PERSIST: return BN_PLAN_FLOW;
    default: return BN_PLAN_AUTO;
    }
}

// Record a BatchNorm call's plan as this thread's last plan.
int record_bn(cudaError_t e, int used) {
    if (e != cudaSuccess) return NRM_ERR_LAUNCH;
    t_last_kind = used;
    t_last_threads = t_last_packs = t_last_stages = t_last_groups = 0;
    return NRM_OK;
}

// ---------------------------------------------------------------------------
// Plan choice for the row operators.
// ---------------------------------------------------------------------------
int round_up_pow2(int64_t v) {
    int r = 1;
    while (r < v && r < (1 << 20)) r <<= 1;
    return r;
}

// Vectorized plans need every row pointer 16-byte aligned and N a multiple of
// the pack width (16 bytes of elements).
int choose_plan(Op op, const RowArgs &a, int dtype, const DevInfo &dev, Plan *plan) {
    const int64_t V = 16 / (int64_t)elem_size(dtype);
    const bool vec_ok = (a.N % V == 0) && aligned(a.x, 16) && aligned(a.y, 16) &&
                        (!a.res || aligned(a.res, 16)) && (!a.res_out || aligned(a.res_out, 16)) &&
                        (!a.p0 || aligned(a.p0, 16)) && (!a.p1 || aligned(a.p1, 16)) &&
                        a.ldx % V == 0 && a.ldy % V == 0 && (!a.res || a.ldr % V == 0) &&
                        (!a.res_out || a.ldro % V == 0);
    const int64_t P = vec_ok ? a.N / V : 0;
    const int64_t kMaxGrid = 0x7fffffff;

    int kind = g_force_kind.load(std::memory_order_relaxed);
    int fthreads = g_force_threads.load(std::memory_order_relaxed);
    int fpacks = g_force_packs.load(std::memory_order_relaxed);
    int fstages = g_force_stages.load(std::memory_order_relaxed);
    int fgroups = g_force_groups.load(std::memory_order_relaxed);

    // Shared-memory stage of the bulk-copy pipeline: one row of x (and one of
    // the residual for add+RMS).
    const int64_t stage_bytes = a.N * (int64_t)elem_size(dtype) * (a.res ? 2 : 1);
    // parameters widened to binary32 in shared memory when they fit in 64 KB
    const int64_t param_bytes = a.N * 4 * (op == OP_LN ? 2 : 1);
    const bool smem_params = param_bytes <= 64 * 1024;
    const int64_t fixed = smem_params ? param_bytes : 0;
    const bool tma_ok = vec_ok && fixed + 2 * stage_bytes <= kSmemMax && P <= 512 * 4;

    // Automatic choice, from measurements on GB300 (cold L2): rows of up to
    // 1024 packs (8192 bf16 / 4096 fp32 values) run fastest as one CTA per row
    // with the row in registers (256 threads x 2 packs at 4096 bf16, 128 x 4
    // for LayerNorm) and the next wave's rows prefetched into L2; rows of
    // up to 2048 packs on persistent CTAs that prefetch the next row (1024 x 2
    // at 16384 bf16); longer rows through the bulk-copy row-group pipeline.
    if (kind == PLAN_AUTO) {
        fthreads = fpacks = fstages = fgroups = 0;
        if (!vec_ok)
            kind = PLAN_GENERIC;
        else if (P <= 32 * 8 && a.rows >= 4 * (int64_t)dev.sms)
            kind = PLAN_WARP;
        else if (P <= 1024)
            kind = PLAN_CTA;
        else if (P <= 2048) {
            // LayerNorm: 4 packs per thread (512 x 4 at 16384 bf16: 13.98 us
            // against 15.64 us for 1024 x 2); the RMS operators keep 2
            kind = PLAN_PERSIST;
            fpacks = op == OP_LN ? 4 : 2;
        } else if (tma_ok) {
            kind = PLAN_TMA;
            fpacks = 4;
            fstages = 2;
        } else if (P <= 1024 * 4)
            kind = PLAN_CTA;
        else
            kind = PLAN_GENERIC;
    }

    Plan p{};
    p.kind = kind;
    p.sms = dev.sms;
    switch (kind) {
    case PLAN_GENERIC: {
        p.threads = fthreads ? fthreads : (a.N >= 4096 ? 512 : 256);
        p.packs = 1;
        p.grid = a.rows < kMaxGrid ? a.rows : kMaxGrid;
        break;
    }
    case PLAN_WARP: {
        if (!vec_ok) return NRM_ERR_UNSUPPORTED;
        int packs = fpacks;
        if (!packs) {
            const int64_t need = (P + 31) / 32;
            packs = need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
        }
        if ((int64_t)packs * 32 < P) return NRM_ERR_UNSUPPORTED;
        p.threads = 128;
        p.packs = packs;
        const int64_t g = (a.rows + 3) / 4;
        p.grid = g < kMaxGrid ? g : kMaxGrid;
        break;
    }
    case PLAN_CTA: {
        if (!vec_ok) return NRM_ERR_UNSUPPORTED;
        int packs = fpacks, threads = fthreads;
        // 128 x 4 for 512 packs for LayerNorm (measured 12.3 us against 14.0 us
        // for 256 x 2 at 4096 x 4096 bf16: half the per-element share of its
        // two row-wide sums) and RMSNorm (2048 x 4096 fp16: 5.65 us against
        // 5.94 us: twice the bytes in flight per thread); add+RMSNorm, with
        // two inputs in flight, keeps 256 x 2
        if (!packs) packs = P <= 256 ? 1 : (op != OP_ADD_RMS && P <= 512) ? 4 : P <= 1024 ? 2 : 4;
        if (!threads) {
            threads = round_up_pow2((P + packs - 1) / packs);
            if (threads < 128) threads = 128;
        }
        if (threads > 1024 || (int64_t)threads * packs < P) return NRM_ERR_UNSUPPORTED;
        p.threads = threads;
        p.packs = packs;
        p.grid = a.rows < kMaxGrid ? a.rows : kMaxGrid;
        // L2 prefetch distance in waves (forced `stages`: 1 = off, s >= 2 = s - 1)
        p.prefetch = fstages == 0 ? 1 : fstages - 1;
        p.stages = fstages;
        break;
    }
    case PLAN_WRAW: {
        // one warp per row: 32 lanes x packs >= P; 8 warps per CTA by default
        if (!vec_ok) return NRM_ERR_UNSUPPORTED;
        int packs = fpacks, threads = fthreads ? fthreads : 256;
        if (!packs) {
            const int64_t need = (P + 31) / 32;
            packs = need <= 4 ? 4 : need <= 8 ? 8 : need <= 16 ? 16 : 32;
        }
        if ((int64_t)packs * 32 < P) return NRM_ERR_UNSUPPORTED;
        p.threads = threads;
        p.packs = packs;
        p.smem_params = smem_params ? 1 : 0;
        p.prefetch = fstages == 0 ? 1 : fstages - 1;  // as the CTA plan
        p.stages = fstages;
        break;
    }
    case PLAN_PERSIST: {
        if (!vec_ok) return NRM_ERR_UNSUPPORTED;
        int packs = fpacks, threads = fthreads;
        if (!packs) packs = P <= 256 ? 1 : P <= 1024 ? 2 : 4;
        if (!threads) {
            threads = round_up_pow2((P + packs - 1) / packs);
            if (threads < 128) threads = 128;
        }
        if (threads > 1024 || (int64_t)threads * packs < P) return NRM_ERR_UNSUPPORTED;
        p.threads = threads;
        p.packs = packs;
        p.smem_params = smem_params ? 1 : 0;
        // L2 prefetch distance in waves (forced `stages`: 1 = off, s >= 2 = s - 1)
        p.prefetch = fstages == 0 ? 1 : fstages - 1;
        p.stages = fstages;
        break;
    }
    case PLAN_CLUSTER: {
        // one row over a cluster of CS CTAs (p.groups), each a contiguous
        // slice of S = P / CS packs held as THREADS x PACKS
        if (!vec_ok) return NRM_ERR_UNSUPPORTED;
        const int cs = fgroups ? fgroups : (P >= 2048 ? 4 : 2);
        if ((cs != 2 && cs != 4 && cs != 8) || P % cs) return NRM_ERR_UNSUPPORTED;
        const int64_t S = P / cs;
        int packs = fpacks, threads = fthreads ? fthreads : 128;
        if (!packs) packs = S <= 128 ? 1 : S <= 256 ? 2 : 4;
        if ((int64_t)threads * packs < S) return NRM_ERR_UNSUPPORTED;
        p.threads = threads;
        p.packs = packs;
        p.groups = cs;
        p.grid = (a.rows < kMaxGrid / cs ? a.rows : kMaxGrid / cs) * cs;
        break;
    }
    case PLAN_TMA: {
        // Row groups of GT threads x PACKS packs (4 preferred), as many groups
        // per CTA as fit in 1024 threads and the shared memory with 3 (else 2)
        // stages each.
        if (!tma_ok) return NRM_ERR_UNSUPPORTED;
        int packs = fpacks, threads = fthreads;
        if (!threads) {
            threads = round_up_pow2((P + 3) / 4);
            threads = threads < 128 ? 128 : threads > 512 ? 512 : threads;
        }
        if (!packs) packs = (int)((P + threads - 1) / threads) <= 2 && threads == 256 ? 2
                            : (P + threads - 1) / threads <= 4 ? 4 : 8;
        if ((int64_t)threads * packs < P) return NRM_ERR_UNSUPPORTED;
        int stages = fstages, groups = fgroups;
        // parameters: binary32 in shared memory when four or more groups share
        // them, else raw packs in shared memory when they fit beside the
        // stages, else through L1 (read through L1, they miss once the stages
        // leave L1 little room: LayerNorm 1024 x 16384 bf16, one 512 x 4 group,
        // 5 stages 25.6 -> 22.6 us with raw packs in shared memory)
        const int64_t raw_bytes = a.N * (int64_t)elem_size(dtype) * (op == OP_LN ? 2 : 1);
        auto params_mode = [&](int gr, int st) {
            const int64_t ring = (int64_t)gr * st * stage_bytes;
            return (smem_params && gr >= 4) ? 1 : raw_bytes + ring <= kSmemMax ? 2 : 0;
        };
        auto fits = [&](int gr, int st) {
            const int m = params_mode(gr, st);
            const int64_t prm = m == 1 ? param_bytes : m == 2 ? raw_bytes : 0;
            return gr * threads <= 1024 && prm + (int64_t)gr * st * stage_bytes <= kSmemMax;
        };
        if (!groups || !stages) {
            int best_g = 0, best_s = 0;
            for (int st : {3, 2}) {
                if (stages && st != stages) continue;
                for (int gr : {8, 4, 2, 1}) {
                    if (groups && gr != groups) continue;
                    if (fits(gr, st) && gr * threads > best_g * threads) {
                        best_g = gr;
                        best_s = st;
                    }
                }
                if (best_g && !stages) break;
            }
            if (!best_g && stages && !groups) {
                for (int gr : {8, 4, 2, 1})
                    if (fits(gr, stages)) { best_g = gr; best_s = stages; break; }
            }
            groups = groups ? groups : best_g;
            stages = stages ? stages : best_s;
        }
        if (groups < 1 || stages < 2 || stages > kMaxStages || !fits(groups, stages))
            return NRM_ERR_UNSUPPORTED;
        p.threads = threads;
        p.packs = packs;
        p.stages = stages;
        p.groups = groups;
        p.smem_params = params_mode(groups, stages);
        break;
    }
    default:
        return NRM_ERR_UNSUPPORTED;
    }
    *plan = p;
    return NRM_OK;
}

// Plan choice for the row softmax: one CTA per row with the row in
// registers while it fits 1024 threads x 4 packs, else the generic plan.
int choose_softmax_plan(const RowArgs &a, int dtype, const DevInfo &dev, Plan *plan) {
    const int64_t V = 16 / (int64_t)elem_size(dtype);
    const bool vec_ok = (a.N % V == 0) && aligned(a.x, 16) && aligned(a.y, 16) &&
                        a.ldx % V == 0 && a.ldy % V == 0;
    const int64_t P = vec_ok ? a.N / V : 0;
    const int64_t kMaxGrid = 0x7fffffff;
    int kind = g_force_kind.load(std::memory_order_relaxed);
    int threads = g_force_threads.load(std::memory_order_relaxed);
    int packs = g_force_packs.load(std::memory_order_relaxed);
    const int fstages = g_force_stages.load(std::memory_order_relaxed);
    if (kind == PLAN_AUTO) {
        threads = packs = 0;
        kind = (vec_ok && P <= 4096) ? PLAN_CTA : PLAN_GENERIC;
    }
    Plan p{};
    p.kind = kind;
    p.sms = dev.sms;
    p.grid = a.rows < kMaxGrid ? a.rows : kMaxGrid;
    if (kind == PLAN_GENERIC) {
        p.threads = threads ? threads : (a.N >= 4096 ? 512 : 256);
        p.packs = 1;
    } else if (kind == PLAN_CTA) {
        if (!vec_ok) return NRM_ERR_UNSUPPORTED;
        if (!threads || !packs) {
            threads = P <= 128 ? 128 : P <= 256 ? 256 : P <= 512 ? 128 : P <= 1024 ? 256
                      : P <= 2048 ? 512 : 1024;
            packs = P <= 256 ? 1 : 4;
        }
        if ((int64_t)threads * packs < P) return NRM_ERR_UNSUPPORTED;
        p.threads = threads;
        p.packs = packs;
        p.prefetch = fstages == 0 ? 1 : fstages - 1;
        p.stages = fstages;
    } else if (kind == PLAN_CLUSTER) {
        // one row over a cluster of CS CTAs (p.groups), as the norms' plan
        if (!vec_ok) return NRM_ERR_UNSUPPORTED;
        const int fgroups = g_force_groups.load(std::memory_order_relaxed);
        const int cs = fgroups ? fgroups : 4;
        if ((cs != 2 && cs != 4 && cs != 8) || P % cs) return NRM_ERR_UNSUPPORTED;
        const int64_t S = P / cs;
        if (!threads) threads = 128;
        if (!packs) packs = S <= 128 ? 1 : S <= 256 ? 2 : 4;
        if ((int64_t)threads * packs < S) return NRM_ERR_UNSUPPORTED;
        p.threads = threads;
        p.packs = packs;
        p.groups = cs;
        p.grid = (a.rows < kMaxGrid / cs ? a.rows : kMaxGrid / cs) * cs;
    } else {
        return NRM_ERR_UNSUPPORTED;
    }
    *plan = p;
    return NRM_OK;
}

int run_row(Op op, RowArgs a, int dtype, cudaStream_t stream) {
    DevInfo dev;
    int st = device_info(&dev);
    if (st != NRM_OK) return st;
    a.fault = fault_word();
    a.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
    a.fN = (float)a.N;
    a.invN = 1.0f / a.fN;
    Plan plan;
    st = op == OP_SOFTMAX ? choose_softmax_plan(a, dtype, dev, &plan)
                          : choose_plan(op, a, dtype, dev, &plan);
    if (st != NRM_OK) return st;
    cudaError_t e;
    switch (op) {
    case OP_LN: e = launch_ln(a, plan, dtype, stream); break;
    case OP_RMS: e = launch_rms(a, plan, dtype, stream); break;
    case OP_SOFTMAX: e = launch_softmax(a, plan, dtype, stream); break;
    default: e = launch_add_rms(a, plan, dtype, stream); break;
    }
    if (e == cudaErrorInvalidConfiguration) {
        cudaGetLastError();
        return NRM_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return NRM_ERR_LAUNCH;
    t_last_kind = plan.kind;
    t_last_threads = plan.threads;
    t_last_packs = plan.packs;
    t_last_stages = plan.stages;
    t_last_groups = plan.groups;
    return NRM_OK;
}

// Shared validation of the row operators: extents, type, eps.
int validate_rows(int64_t rows, int64_t N, float eps, int dtype) {
    if (!dtype_ok(dtype)) return NRM_ERR_DTYPE;
    if (rows < 0 || N < 1) return NRM_ERR_SHAPE;
    const size_t es = elem_size(dtype);
    if (rows > 0 && (uint64_t)N > (uint64_t)INT64_MAX / (uint64_t)rows / es) return NRM_ERR_SHAPE;
    if (!eps_ok(eps)) return NRM_ERR_VALUE;
    return NRM_OK;
}

// Row strides: at least N (rows must not overlap) and small enough that the
// last row's end fits a 64-bit byte offset.
int validate_ld(int64_t rows, int64_t N, size_t es, std::initializer_list<int64_t> lds) {
    for (int64_t ld : lds) {
        if (ld < N) return NRM_ERR_SHAPE;
        if ((uint64_t)ld > (uint64_t)INT64_MAX / (uint64_t)rows / es) return NRM_ERR_SHAPE;
    }
    return NRM_OK;
}

// A strided 2-D extent in bytes: `rows` rows of `width` bytes, `ld` bytes
// apart (a contiguous vector is one row).
struct RSpan {
    uintptr_t base = 0;
    int64_t ld = 0, width = 0, rows = 0;
    bool live() const { return base && width > 0 && rows > 0; }
    uintptr_t end() const { return base + (uintptr_t)((rows - 1) * ld + width); }
};
RSpan rspan(const void *p, int64_t ld_elems, int64_t rows, int64_t width_elems, size_t es) {
    RSpan s;
    if (p && rows > 0) {
        s.base = reinterpret_cast<uintptr_t>(p);
        s.ld = ld_elems * (int64_t)es;
        s.width = width_elems * (int64_t)es;
        s.rows = rows;
    }
    return s;
}

int64_t floor_div(int64_t a, int64_t b) {  // b > 0
    const int64_t q = a / b;
    return (a % b != 0 && a < 0) ? q - 1 : q;
}

// Whether two extents share a byte.  Two extents with the same row stride and
// row count (columns of one padded buffer, for instance) are tested exactly:
// rows i of A and j of B meet iff for k = j - i, d + k*ld lies in
// (-width_b, width_a), d = base_b - base_a.  Anything else is compared by its
// outer bounds (conservative).
bool roverlap(const RSpan &a, const RSpan &b) {
    if (!a.live() || !b.live()) return false;
    if (!(a.base < b.end() && b.base < a.end())) return false;
    if (a.rows == 1 || b.rows == 1 || a.ld != b.ld || a.rows != b.rows) return true;
    const int64_t d = (int64_t)(b.base - a.base);  // two's complement difference
    const int64_t L = a.ld;
    int64_t k = floor_div(-b.width - d, L) + 1;    // smallest k with d + k*L > -width_b
    if (k < -(a.rows - 1)) k = -(a.rows - 1);
    return k <= a.rows - 1 && d + k * L < a.width;
}

int check_elem_alignment(std::initializer_list<const void *> ps, size_t es) {
    for (const void *p : ps)
        if (p && !aligned(p, es)) return NRM_ERR_VALUE;
    return NRM_OK;
}

}  // namespace

namespace nrm {
size_t bn_group_bytes() { return g_bn_group_bytes.load(std::memory_order_relaxed); }
}  // namespace nrm

extern "C" {

int ln_fwd_ld(const void *x, int64_t ldx, const void *gamma, const void *beta, void *y,
              int64_t ldy, float *mean, float *rstd, int64_t rows, int64_t N, float eps, int dtype,
              cudaStream_t stream) {
    int st = validate_rows(rows, N, eps, dtype);
    if (st != NRM_OK) return st;
    if (rows == 0) return NRM_OK;  // empty input: no pointer is used
    if (!x || !y) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = validate_ld(rows, N, es, {ldx, ldy})) != NRM_OK) return st;
    if ((st = check_elem_alignment({x, gamma, beta, y}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({mean, rstd}, 4)) != NRM_OK) return st;
    const RSpan sx = rspan(x, ldx, rows, N, es), sy = rspan(y, ldy, rows, N, es),
                sg = rspan(gamma, N, 1, N, es), sb = rspan(beta, N, 1, N, es),
                sm = rspan(mean, rows, 1, rows, 4), sr = rspan(rstd, rows, 1, rows, 4);
    for (const RSpan &o : {sy, sm, sr})
        for (const RSpan &i : {sx, sg, sb})
            if (roverlap(o, i)) return NRM_ERR_ALIAS;
    if (roverlap(sy, sm) || roverlap(sy, sr) || roverlap(sm, sr)) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, gamma, beta, y, mean, rstd})) != NRM_OK) return st;
    RowArgs a{x, nullptr, gamma, beta, nullptr, y, mean, rstd, rows, N, eps, nullptr, 0, 0.f, 0.f,
              ldx, N, N, ldy};
    return run_row(OP_LN, a, dtype, stream);
}

int ln_fwd(const void *x, const void *gamma, const void *beta, void *y, float *mean,
           float *rstd, int64_t rows, int64_t N, float eps, int dtype, cudaStream_t stream) {
    return ln_fwd_ld(x, N, gamma, beta, y, N, mean, rstd, rows, N, eps, dtype, stream);
}

int rms_fwd_ld(const void *x, int64_t ldx, const void *w, void *y, int64_t ldy, float *rstd,
               int64_t rows, int64_t N, float eps, int dtype, cudaStream_t stream) {
    int st = validate_rows(rows, N, eps, dtype);
    if (st != NRM_OK) return st;
    if (rows == 0) return NRM_OK;  // empty input: no pointer is used
    if (!x || !y) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = validate_ld(rows, N, es, {ldx, ldy})) != NRM_OK) return st;
    if ((st = check_elem_alignment({x, w, y}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({rstd}, 4)) != NRM_OK) return st;
    const RSpan sx = rspan(x, ldx, rows, N, es), sy = rspan(y, ldy, rows, N, es),
                sw = rspan(w, N, 1, N, es), sr = rspan(rstd, rows, 1, rows, 4);
    for (const RSpan &o : {sy, sr})
        for (const RSpan &i : {sx, sw})
            if (roverlap(o, i)) return NRM_ERR_ALIAS;
    if (roverlap(sy, sr)) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, w, y, rstd})) != NRM_OK) return st;
    RowArgs a{x, nullptr, w, nullptr, nullptr, y, nullptr, rstd, rows, N, eps, nullptr, 0, 0.f, 0.f,
              ldx, N, N, ldy};
    return run_row(OP_RMS, a, dtype, stream);
}

int rms_fwd(const void *x, const void *w, void *y, float *rstd, int64_t rows, int64_t N,
            float eps, int dtype, cudaStream_t stream) {
    return rms_fwd_ld(x, N, w, y, N, rstd, rows, N, eps, dtype, stream);
}

int add_rms_fwd_ld(const void *x, int64_t ldx, const void *residual, int64_t ldr, const void *w,
                   void *residual_out, int64_t ldro, void *y, int64_t ldy, float *rstd,
                   int64_t rows, int64_t N, float eps, int dtype, cudaStream_t stream) {
    int st = validate_rows(rows, N, eps, dtype);
    if (st != NRM_OK) return st;
    if (rows == 0) return NRM_OK;  // empty input: no pointer is used
    if (!x || !residual || !residual_out || !y) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = validate_ld(rows, N, es, {ldx, ldr, ldro, ldy})) != NRM_OK) return st;
    if ((st = check_elem_alignment({x, residual, w, residual_out, y}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({rstd}, 4)) != NRM_OK) return st;
    const RSpan sx = rspan(x, ldx, rows, N, es), sres = rspan(residual, ldr, rows, N, es),
                sw = rspan(w, N, 1, N, es), sro = rspan(residual_out, ldro, rows, N, es),
                sy = rspan(y, ldy, rows, N, es), sr = rspan(rstd, rows, 1, rows, 4);
    // residual_out may be exactly residual, with the same row stride (the
    // residual stream updated in place)
    const bool inplace = residual_out == residual && ldro == ldr;
    for (const RSpan &i : {sx, sw})
        for (const RSpan &o : {sro, sy, sr})
            if (roverlap(o, i)) return NRM_ERR_ALIAS;
    if (!inplace && roverlap(sro, sres)) return NRM_ERR_ALIAS;
    if (roverlap(sy, sres) || roverlap(sr, sres)) return NRM_ERR_ALIAS;
    if (roverlap(sro, sy) || roverlap(sro, sr) || roverlap(sy, sr)) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, residual, w, residual_out, y, rstd})) != NRM_OK) return st;
    RowArgs a{x, residual, w, nullptr, residual_out, y, nullptr, rstd, rows, N, eps, nullptr, 0,
              0.f, 0.f, ldx, ldr, ldro, ldy};
    return run_row(OP_ADD_RMS, a, dtype, stream);
}

int add_rms_fwd(const void *x, const void *residual, const void *w, void *residual_out, void *y,
                float *rstd, int64_t rows, int64_t N, float eps, int dtype, cudaStream_t stream) {
    return add_rms_fwd_ld(x, N, residual, N, w, residual_out, N, y, N, rstd, rows, N, eps, dtype,
                          stream);
}

int softmax_fwd_ld(const void *x, int64_t ldx, void *y, int64_t ldy, float *row_max,
                   float *row_sum, int64_t rows, int64_t N, int dtype, cudaStream_t stream) {
    int st = validate_rows(rows, N, 0.f, dtype);
    if (st != NRM_OK) return st;
    if (rows == 0) return NRM_OK;  // empty input: no pointer is used
    if (!x || !y) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = validate_ld(rows, N, es, {ldx, ldy})) != NRM_OK) return st;
    if ((st = check_elem_alignment({x, y}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({row_max, row_sum}, 4)) != NRM_OK) return st;
    const RSpan sx = rspan(x, ldx, rows, N, es), sy = rspan(y, ldy, rows, N, es),
                sm = rspan(row_max, rows, 1, rows, 4), ss = rspan(row_sum, rows, 1, rows, 4);
    for (const RSpan &o : {sy, sm, ss})
        if (roverlap(o, sx)) return NRM_ERR_ALIAS;
    if (roverlap(sy, sm) || roverlap(sy, ss) || roverlap(sm, ss)) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, y, row_max, row_sum})) != NRM_OK) return st;
    RowArgs a{x, nullptr, nullptr, nullptr, nullptr, y, row_max, row_sum, rows, N, 0.f,
              nullptr, 0, 0.f, 0.f, ldx, N, N, ldy};
    return run_row(OP_SOFTMAX, a, dtype, stream);
}

int softmax_fwd(const void *x, void *y, float *row_max, float *row_sum, int64_t rows, int64_t N,
                int dtype, cudaStream_t stream) {
    return softmax_fwd_ld(x, N, y, N, row_max, row_sum, rows, N, dtype, stream);
}

size_t bn_fwd_train_workspace_size(int64_t batch, int64_t C, int64_t HW, int dtype) {
    if (!dtype_ok(dtype) || batch < 1 || C < 1 || HW < 1) return 0;
    // 8 bytes per chunk of at most 1024 packs of a plane (the streaming and
    // one-pass plans; the scalar plan needs one per plane, never more), then
    // the one-pass plan's per-channel statistics and control words
    const int64_t V = 16 / (int64_t)elem_size(dtype);
    const int64_t packs = (HW + V - 1) / V;
    const int64_t nch = (packs + kBnChunkPacks - 1) / kBnChunkPacks;
    if ((uint64_t)batch > (uint64_t)INT64_MAX / 16 / (uint64_t)C / (uint64_t)nch) return 0;
    return bn_flow_ws_bytes(C, batch * C * nch);
}

}  // extern "C"

namespace {

// The BatchNorm training forward behind both entry points: bn_fwd_train
// (caller workspace) and bn_fwd_train_noalloc (fixed == true: the library's
// fixed partials array, bn_fixed_workspace in bn.cu).  Same validation, plan
// choice, wait limit and plan record for both.
int bn_train_call(const void *x, const void *gamma, const void *beta, void *y, float *save_mean,
                  float *save_rstd, float *running_mean, float *running_var, int64_t batch,
                  int64_t C, int64_t HW, float eps, float momentum, int dtype, void *workspace,
                  size_t workspace_bytes, bool fixed, cudaStream_t stream) {
    if (!dtype_ok(dtype)) return NRM_ERR_DTYPE;
    if (batch < 1 || C < 1 || HW < 1) return NRM_ERR_SHAPE;
    const size_t es = elem_size(dtype);
    if ((uint64_t)batch > (uint64_t)INT64_MAX / (uint64_t)C / (uint64_t)HW / es)
        return NRM_ERR_SHAPE;
    if (batch * HW < 2) return NRM_ERR_SHAPE;
    if (fixed && batch * C > kBnFixedPlanes) return NRM_ERR_TOO_LARGE;
    if (!eps_ok(eps) || !(momentum >= 0.f && momentum <= 1.f)) return NRM_ERR_VALUE;
    if (!x || !y) return NRM_ERR_NULL;
    int st;
    if ((st = check_elem_alignment({x, gamma, beta, y}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({save_mean, save_rstd, running_mean, running_var}, 4)) != NRM_OK)
        return st;
    const size_t need = fixed ? 0 : bn_fwd_train_workspace_size(batch, C, HW, dtype);
    if (!fixed && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return NRM_ERR_WORKSPACE;
    const size_t tb = (size_t)batch * (size_t)C * (size_t)HW * es;
    const Span sx = span(x, tb), sy = span(y, tb), sg = span(gamma, C * es), sb = span(beta, C * es),
               ssm = span(save_mean, C * 4), ssr = span(save_rstd, C * 4),
               srm = span(running_mean, C * 4), srv = span(running_var, C * 4),
               sws = span(fixed ? nullptr : workspace, need);
    const Span outs[] = {sy, ssm, ssr, srm, srv, sws};
    const Span ins[] = {sx, sg, sb};
    for (const Span &o : outs)
        for (const Span &i : ins)
            if (overlap(o, i)) return NRM_ERR_ALIAS;
    for (int i = 0; i < 6; ++i)
        for (int j = i + 1; j < 6; ++j)
            if (overlap(outs[i], outs[j])) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, gamma, beta, y, save_mean, save_rstd, running_mean, running_var,
                              fixed ? nullptr : workspace})) != NRM_OK)
        return st;
    DevInfo dev;
    if ((st = device_info(&dev)) != NRM_OK) return st;
    if (fixed && (st = bn_fixed_workspace(&workspace, &workspace_bytes)) != NRM_OK) return st;
    int bn_plan = bn_plan_from_forced();
    if (fixed) {
        // the streaming plan keeps one partial per chunk of at most
        // kBnChunkPacks packs; when those do not fit the fixed array, the
        // other plans (per-plane partials, or none) still do
        const int64_t V = 16 / (int64_t)es;
        const int64_t nch = ((HW + V - 1) / V + kBnChunkPacks - 1) / kBnChunkPacks;
        if (batch * C * nch > kBnFixedPlanes &&
            (bn_plan == BN_PLAN_AUTO || bn_plan == BN_PLAN_STREAM))
            bn_plan = BN_PLAN_NO_STREAM;
    }
    BnArgs a{x, gamma, beta, y, save_mean, save_rstd, running_mean, running_var, batch, C, HW,
             eps, momentum, workspace, fault_word(), g_wait_limit.load(std::memory_order_relaxed),
             bn_plan, workspace_bytes, 0, 0};
    if (g_force_kind.load(std::memory_order_relaxed) == PLAN_PERSIST) {
        a.prefetch = g_force_stages.load(std::memory_order_relaxed);
        a.packs = g_force_packs.load(std::memory_order_relaxed);
    }
    if (g_force_kind.load(std::memory_order_relaxed) == PLAN_TMA) {
        a.cluster_size = g_force_stages.load(std::memory_order_relaxed);
        a.max_clusters = g_force_threads.load(std::memory_order_relaxed);
    }
    int used = 0;
    return record_bn(launch_bn_train(a, dtype, dev.sms, stream, &used), used);
}

}  // namespace

extern "C" {

int bn_fwd_train(const void *x, const void *gamma, const void *beta, void *y, float *save_mean,
                 float *save_rstd, float *running_mean, float *running_var, int64_t batch,
                 int64_t C, int64_t HW, float eps, float momentum, int dtype, void *workspace,
                 size_t workspace_bytes, cudaStream_t stream) {
    return bn_train_call(x, gamma, beta, y, save_mean, save_rstd, running_mean, running_var, batch,
                         C, HW, eps, momentum, dtype, workspace, workspace_bytes, false, stream);
}

// No page has this entry point: bn_fwd_train for callers that cannot allocate
// device memory when they call (the header says who and why).  The partials
// live in the library's fixed array (bn.cu).
int bn_fwd_train_noalloc(const void *x, const void *gamma, const void *beta, void *y,
                         float *save_mean, float *save_rstd, float *running_mean,
                         float *running_var, int64_t batch, int64_t C, int64_t HW, float eps,
                         float momentum, int dtype, cudaStream_t stream) {
    return bn_train_call(x, gamma, beta, y, save_mean, save_rstd, running_mean, running_var, batch,
                         C, HW, eps, momentum, dtype, nullptr, 0, true, stream);
}

int bn_fwd_infer(const void *x, const void *gamma, const void *beta, void *y,
                 const float *running_mean, const float *running_var, int64_t batch, int64_t C,
                 int64_t HW, float eps, int dtype, cudaStream_t stream) {
    if (!dtype_ok(dtype)) return NRM_ERR_DTYPE;
    if (batch < 0 || C < 1 || HW < 1) return NRM_ERR_SHAPE;
    const size_t es = elem_size(dtype);
    if (batch > 0 && (uint64_t)batch > (uint64_t)INT64_MAX / (uint64_t)C / (uint64_t)HW / es)
        return NRM_ERR_SHAPE;
    if (!eps_ok(eps)) return NRM_ERR_VALUE;
    if (batch == 0) return NRM_OK;  // empty batch: no pointer is used
    if (!x || !y || !running_mean || !running_var) return NRM_ERR_NULL;
    int st;
    if ((st = check_elem_alignment({x, gamma, beta, y}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({running_mean, running_var}, 4)) != NRM_OK) return st;
    const size_t tb = (size_t)batch * (size_t)C * (size_t)HW * es;
    const Span sy = span(y, tb);
    for (const Span &i : {span(x, tb), span(gamma, C * es), span(beta, C * es),
                          span(running_mean, C * 4), span(running_var, C * 4)})
        if (overlap(sy, i)) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, gamma, beta, y, running_mean, running_var})) != NRM_OK) return st;
    DevInfo dev;
    if ((st = device_info(&dev)) != NRM_OK) return st;
    BnInferArgs a{x, gamma, beta, y, running_mean, running_var, batch, C, HW, eps,
                  bn_plan_from_forced()};
    int used = 0;
    return record_bn(launch_bn_infer(a, dtype, dev.sms, stream, &used), used);
}

size_t bn_bwd_workspace_size(int64_t batch, int64_t C, int64_t HW, int dtype) {
    return bn_fwd_train_workspace_size(batch, C, HW, dtype);
}

int bn_bwd(const void *dy, const void *x, const void *gamma, const float *save_mean,
           const float *save_rstd, void *dx, float *dgamma, float *dbeta, int64_t batch,
           int64_t C, int64_t HW, int dtype, void *workspace, size_t workspace_bytes,
           cudaStream_t stream) {
    if (!dtype_ok(dtype)) return NRM_ERR_DTYPE;
    if (batch < 1 || C < 1 || HW < 1) return NRM_ERR_SHAPE;
    const size_t es = elem_size(dtype);
    if ((uint64_t)batch > (uint64_t)INT64_MAX / (uint64_t)C / (uint64_t)HW / es)
        return NRM_ERR_SHAPE;
    if (!dy || !x || !save_mean || !save_rstd || !dx) return NRM_ERR_NULL;
    int st;
    if ((st = check_elem_alignment({dy, x, gamma, dx}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({save_mean, save_rstd, dgamma, dbeta}, 4)) != NRM_OK) return st;
    const size_t need = bn_bwd_workspace_size(batch, C, HW, dtype);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return NRM_ERR_WORKSPACE;
    const size_t tb = (size_t)batch * (size_t)C * (size_t)HW * es;
    const Span outs[] = {span(dx, tb), span(dgamma, C * 4), span(dbeta, C * 4),
                         span(workspace, need)};
    const Span ins[] = {span(dy, tb), span(x, tb), span(gamma, C * es), span(save_mean, C * 4),
                        span(save_rstd, C * 4)};
    for (const Span &o : outs)
        for (const Span &i : ins)
            if (overlap(o, i)) return NRM_ERR_ALIAS;
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (overlap(outs[i], outs[j])) return NRM_ERR_ALIAS;
    if ((st = check_pointers({dy, x, gamma, save_mean, save_rstd, dx, dgamma, dbeta,
                              workspace})) != NRM_OK)
        return st;
    DevInfo dev;
    if ((st = device_info(&dev)) != NRM_OK) return st;
    BnBwdArgs a{dy, x, gamma, save_mean, save_rstd, dx, dgamma, dbeta, batch, C, HW, workspace,
                bn_plan_from_forced(), fault_word(), g_wait_limit.load(std::memory_order_relaxed),
                workspace_bytes, 0};
    if (g_force_kind.load(std::memory_order_relaxed) == PLAN_PERSIST)
        a.prefetch = g_force_stages.load(std::memory_order_relaxed);
    int used = 0;
    return record_bn(launch_bn_bwd(a, dtype, dev.sms, stream, &used), used);
}

// ---------------------------------------------------------------------------
// Synchronized BatchNorm pieces.
// ---------------------------------------------------------------------------
namespace {
int bn_sync_shape(int64_t batch, int64_t C, int64_t HW, int dtype) {
    if (!dtype_ok(dtype)) return NRM_ERR_DTYPE;
    if (batch < 1 || C < 1 || HW < 1) return NRM_ERR_SHAPE;
    if ((uint64_t)batch > (uint64_t)INT64_MAX / (uint64_t)C / (uint64_t)HW / 8) return NRM_ERR_SHAPE;
    return NRM_OK;
}
}  // namespace

int bn_fwd_partial_stats(const void *x, double *stats, int64_t batch, int64_t C, int64_t HW,
                         int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    int st = bn_sync_shape(batch, C, HW, dtype);
    if (st != NRM_OK) return st;
    if (!x || !stats) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = check_elem_alignment({x}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({stats}, 8)) != NRM_OK) return st;
    const size_t need = bn_fwd_train_workspace_size(batch, C, HW, dtype);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return NRM_ERR_WORKSPACE;
    const Span sx = span(x, (size_t)batch * C * HW * es), ss = span(stats, (size_t)C * 24),
               sw = span(workspace, need);
    if (overlap(ss, sx) || overlap(sw, sx) || overlap(ss, sw)) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, stats, workspace})) != NRM_OK) return st;
    DevInfo dev;
    if ((st = device_info(&dev)) != NRM_OK) return st;
    BnArgs a{x, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, batch, C, HW, 0.f,
             0.f, workspace, nullptr, 0, BN_PLAN_SCALAR};
    const int64_t V = 16 / (int64_t)es;
    const float2 *ws = static_cast<const float2 *>(workspace);
    cudaError_t e;
    int used;
    // the cluster plan in statistics-only mode: one launch, x read once, the
    // channel's statistics folded over the cluster (binary32, shifted by
    // x[0, c, 0]) and written in binary64; else the streaming units and a
    // binary64 fold
    const int forced = g_force_kind.load(std::memory_order_relaxed);
    if (forced == PLAN_AUTO || forced == PLAN_TMA) {
        BnArgs ac = a;
        ac.fault = fault_word();
        ac.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
        ac.stats_out = stats;
        if (forced == PLAN_TMA) ac.cluster_size = g_force_stages.load(std::memory_order_relaxed);
        bool launched = false;
        e = launch_bn_cluster_stats(ac, dtype, stream, &launched);
        if (launched || e != cudaSuccess) return record_bn(e, PLAN_TMA);
    }
    if (HW % V == 0 && aligned(x, 16) && HW / V < kBnUnitPlaneLimit) {
        int nch = 0, cpk = 0, q = 0;
        e = launch_bn_unit_stats_host(a, dtype, dev.sms, stream, &nch, &cpk, &q);
        if (e == cudaSuccess)
            e = launch_bn_fold_stats(ws, x, stats, batch * nch, C, HW, nch, cpk, q, (int)V, dtype,
                                     stream);
        used = PLAN_CTA;
    } else {
        e = launch_bn_plane_stats(a, dtype, dev.sms, stream);
        if (e == cudaSuccess)
            e = launch_bn_fold_stats(ws, x, stats, batch, C, HW, 1, 0, 0, 0, dtype, stream);
        used = PLAN_GENERIC;
    }
    return record_bn(e, used);
}

int bn_fwd_apply_stats(const void *x, const void *gamma, const void *beta, void *y,
                       const double *parts, int64_t nparts, float *save_mean, float *save_rstd,
                       float *running_mean, float *running_var, int64_t batch, int64_t C,
                       int64_t HW, float eps, float momentum, int dtype, cudaStream_t stream) {
    int st = bn_sync_shape(batch, C, HW, dtype);
    if (st != NRM_OK) return st;
    if (nparts < 1 || (uint64_t)nparts > (uint64_t)INT64_MAX / 24 / (uint64_t)C) return NRM_ERR_SHAPE;
    if (!eps_ok(eps) || !(momentum >= 0.f && momentum <= 1.f)) return NRM_ERR_VALUE;
    if (!x || !y || !parts) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = check_elem_alignment({x, gamma, beta, y}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({save_mean, save_rstd, running_mean, running_var}, 4)) != NRM_OK)
        return st;
    if ((st = check_elem_alignment({parts}, 8)) != NRM_OK) return st;
    const size_t tb = (size_t)batch * C * HW * es, cb = (size_t)C * 4;
    const Span outs[] = {span(y, tb), span(save_mean, cb), span(save_rstd, cb),
                         span(running_mean, cb), span(running_var, cb)};
    const Span ins[] = {span(x, tb), span(gamma, C * es), span(beta, C * es),
                        span(parts, (size_t)nparts * C * 24)};
    for (const Span &o : outs)
        for (const Span &i : ins)
            if (overlap(o, i)) return NRM_ERR_ALIAS;
    for (int i = 0; i < 5; ++i)
        for (int j = i + 1; j < 5; ++j)
            if (overlap(outs[i], outs[j])) return NRM_ERR_ALIAS;
    if ((st = check_pointers({x, gamma, beta, y, parts, save_mean, save_rstd, running_mean,
                              running_var})) != NRM_OK)
        return st;
    DevInfo dev;
    if ((st = device_info(&dev)) != NRM_OK) return st;
    BnSyncArgs a{x, nullptr, gamma, beta, y, nullptr, nullptr, parts, nparts, 0, save_mean,
                 save_rstd, running_mean, running_var, nullptr, nullptr, batch, C, HW, eps,
                 momentum};
    return record_bn(launch_bn_apply_stats(a, dtype, dev.sms, stream), PLAN_GENERIC);
}

int bn_bwd_partial_sums(const void *dy, const void *x, const float *save_mean,
                        const float *save_rstd, double *sums, int64_t batch, int64_t C,
                        int64_t HW, int dtype, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
    int st = bn_sync_shape(batch, C, HW, dtype);
    if (st != NRM_OK) return st;
    if (!dy || !x || !save_mean || !save_rstd || !sums) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = check_elem_alignment({dy, x}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({save_mean, save_rstd}, 4)) != NRM_OK) return st;
    if ((st = check_elem_alignment({sums}, 8)) != NRM_OK) return st;
    const size_t need = bn_bwd_workspace_size(batch, C, HW, dtype);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return NRM_ERR_WORKSPACE;
    const size_t tb = (size_t)batch * C * HW * es;
    const Span outs[] = {span(sums, (size_t)C * 16), span(workspace, need)};
    const Span ins[] = {span(dy, tb), span(x, tb), span(save_mean, C * 4), span(save_rstd, C * 4)};
    for (const Span &o : outs)
        for (const Span &i : ins)
            if (overlap(o, i)) return NRM_ERR_ALIAS;
    if (overlap(outs[0], outs[1])) return NRM_ERR_ALIAS;
    if ((st = check_pointers({dy, x, save_mean, save_rstd, sums, workspace})) != NRM_OK) return st;
    DevInfo dev;
    if ((st = device_info(&dev)) != NRM_OK) return st;
    BnBwdArgs a{dy, x, nullptr, save_mean, save_rstd, nullptr, nullptr, nullptr, batch, C, HW,
                workspace, BN_PLAN_SCALAR};
    const int64_t V = 16 / (int64_t)es;
    const float2 *ws = static_cast<const float2 *>(workspace);
    cudaError_t e;
    int used;
    if (HW % V == 0 && aligned(x, 16) && aligned(dy, 16) && HW / V < kBnUnitPlaneLimit) {
        int nch = 0;
        e = launch_bn_bwd_unit_sums_host(a, dtype, dev.sms, stream, &nch);
        if (e == cudaSuccess) e = launch_bn_fold_sums(ws, save_rstd, sums, batch * nch, C, stream);
        used = PLAN_CTA;
    } else {
        e = launch_bn_bwd_plane_sums(a, dtype, dev.sms, stream);
        if (e == cudaSuccess) e = launch_bn_fold_sums(ws, save_rstd, sums, batch, C, stream);
        used = PLAN_GENERIC;
    }
    return record_bn(e, used);
}

int bn_bwd_apply_sums(const void *dy, const void *x, const void *gamma, const float *save_mean,
                      const float *save_rstd, const double *parts, int64_t nparts, int64_t count,
                      void *dx, float *dgamma, float *dbeta, int64_t batch, int64_t C, int64_t HW,
                      int dtype, cudaStream_t stream) {
    int st = bn_sync_shape(batch, C, HW, dtype);
    if (st != NRM_OK) return st;
    if (nparts < 1 || (uint64_t)nparts > (uint64_t)INT64_MAX / 16 / (uint64_t)C) return NRM_ERR_SHAPE;
    if (count < batch * HW) return NRM_ERR_SHAPE;  // the global count includes this batch
    if (!dy || !x || !save_mean || !save_rstd || !parts || !dx) return NRM_ERR_NULL;
    const size_t es = elem_size(dtype);
    if ((st = check_elem_alignment({dy, x, gamma, dx}, es)) != NRM_OK) return st;
    if ((st = check_elem_alignment({save_mean, save_rstd, dgamma, dbeta}, 4)) != NRM_OK) return st;
    if ((st = check_elem_alignment({parts}, 8)) != NRM_OK) return st;
    const size_t tb = (size_t)batch * C * HW * es;
    const Span outs[] = {span(dx, tb), span(dgamma, C * 4), span(dbeta, C * 4)};
    const Span ins[] = {span(dy, tb), span(x, tb), span(gamma, C * es), span(save_mean, C * 4),
                        span(save_rstd, C * 4), span(parts, (size_t)nparts * C * 16)};
    for (const Span &o : outs)
        for (const Span &i : ins)
            if (overlap(o, i)) return NRM_ERR_ALIAS;
    if (overlap(outs[0], outs[1]) || overlap(outs[0], outs[2]) || overlap(outs[1], outs[2]))
        return NRM_ERR_ALIAS;
    if ((st = check_pointers({dy, x, gamma, save_mean, save_rstd, parts, dx, dgamma, dbeta})) !=
        NRM_OK)
        return st;
    DevInfo dev;
    if ((st = device_info(&dev)) != NRM_OK) return st;
    BnSyncArgs a{x, dy, gamma, nullptr, dx, save_mean, save_rstd, parts, nparts, count, nullptr,
                 nullptr, nullptr, nullptr, dgamma, dbeta, batch, C, HW, 0.f, 0.f};
    return record_bn(launch_bn_apply_sums(a, dtype, dev.sms, stream), PLAN_GENERIC);
}

const char *nrm_status_string(int status) {
    switch (status) {
    case NRM_OK: return "ok";
    case NRM_ERR_NULL: return "a required pointer is NULL";
    case NRM_ERR_SHAPE: return "invalid shape (negative extent, N < 1, size overflow, or BatchNorm count < 2)";
    case NRM_ERR_DTYPE: return "unknown dtype";
    case NRM_ERR_ALIAS: return "an output overlaps an input or another output";
    case NRM_ERR_VALUE: return "invalid value (eps, momentum, or a pointer not aligned to its element size)";
    case NRM_ERR_UNSUPPORTED: return "not supported for these arguments";
    case NRM_ERR_WORKSPACE: return "workspace missing, too small or not 16-byte aligned";
    case NRM_ERR_DEVICE: return "no usable current CUDA device";
    case NRM_ERR_LAUNCH: return "kernel launch failed";
    case NRM_ERR_POINTER: return "a pointer is not device memory of the current device";
    case NRM_ERR_TOO_LARGE: return "batch * C exceeds the fixed capacity (65536) of bn_fwd_train_noalloc";
    default: return "unknown status";
    }
}

int nrm_force_plan(int plan, int threads, int packs, int stages, int groups) {
    if (plan < NRM_PLAN_AUTO || plan > NRM_PLAN_CLUSTER || threads < 0 || packs < 0 || stages < 0 ||
        stages > kMaxStages || groups < 0 || groups > 15)
        return NRM_ERR_UNSUPPORTED;
    g_force_kind.store(plan);
    g_force_threads.store(plan ? threads : 0);
    g_force_packs.store(plan ? packs : 0);
    g_force_stages.store(plan ? stages : 0);
    g_force_groups.store(plan ? groups : 0);
    return NRM_OK;
}

void nrm_last_plan(int *plan, int *threads, int *packs, int *stages, int *groups) {
    if (plan) *plan = t_last_kind;
    if (threads) *threads = t_last_threads;
    if (packs) *packs = t_last_packs;
    if (stages) *stages = t_last_stages;
    if (groups) *groups = t_last_groups;
}

unsigned nrm_set_wait_limit(unsigned tries) { return g_wait_limit.exchange(tries); }

int nrm_set_pointer_checks(int enable) { return g_pointer_checks.exchange(enable ? 1 : 0); }

size_t nrm_set_bn_group_bytes(size_t bytes) { return g_bn_group_bytes.exchange(bytes); }

}  // extern "C"
