// row_pipe.cuh -- the persistent row-group pipeline (plan NRM_PLAN_TMA).
//
// One CTA per SM (or a few) holds G independent row groups of GT threads.
// Each group streams its rows through its own ring of `stages` shared-memory
// stages: the group leader claims the next row of the CTA's range from a
// shared-memory counter and starts one bulk asynchronous copy per input row
// (cp.async.bulk, completed on the stage's mbarrier), `stages` rows ahead of
// the row the group is reducing.  So loads are always in flight while rows
// are reduced, without holding them in registers, and every CTA gets a
// contiguous, balanced range of rows (its count differs from any other CTA's
// by at most one) that its groups share dynamically.
//
// Per row a group: waits for its stage, copies the row's packs into
// registers (widened to binary32 once when a thread holds at most 4 packs,
// else unpacked again for each pass), releases the stage at the first group
// barrier (the leader starts the next copy into it), and makes two
// (LayerNorm) or one (RMS ops) group-wide sums.  Parameters are read from
// shared memory: widened to binary32 (SmemParams) when several groups share
// them and they fit, else as raw packs (SmemRawParams) when those fit beside
// the stages; else from global memory through L1.
//
// Termination and failure are decided together at the first group barrier
// (bar.red.or): a leader that finds the range exhausted publishes row -1 for
// the stage and arrives on its barrier without a copy; a thread whose bounded
// wait gives up raises the same flag.  Either way every thread of the group
// leaves the loop at the same point, so no named barrier is left waiting.
// After a give-up the leader waits (bounded) for its copies still in flight
// before the CTA releases its shared memory.
//
// Included by row_kernels.cuh inside namespace nrm, after the row sources,
// parameter views and reducers it uses.
#pragma once

template <int OP, typename T>
__device__ __forceinline__ void pipe_claim(const RowArgs &a, unsigned long long *next_row,
                                           int64_t r1, long long *slot_row, uint64_t *full,
                                           unsigned char *ring, uint32_t stage_bytes,
                                           uint32_t row_bytes, const int s) {
    const long long r = (long long)atomicAdd(next_row, 1ULL);
    if (r < r1) {
        slot_row[s] = r;
        unsigned char *dst = ring + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        bulk_g2s(dst, static_cast<const T *>(a.x) + r * a.ldx, row_bytes, &full[s]);
        if (OP == OP_ADD_RMS)
            bulk_g2s(dst + row_bytes, static_cast<const T *>(a.res) + r * a.ldr, row_bytes,
                     &full[s]);
    } else {
        slot_row[s] = -1;
        mbar_arrive(&full[s]);  // completes the phase without data
    }
}

// Launch bounds ask for at least 1024 resident threads per SM (at most 64
// registers per thread), so several CTAs share an SM and their rows overlap.
template <int OP, typename T, int GT, int PACKS, int G>
__global__ void __launch_bounds__(GT *G, (1024 / (GT * G)) > 0 ? (1024 / (GT * G)) : 1)
    row_pipe_kernel(const RowArgs a, const int stages, const int smem_params) {
    using io2 = IO2<T>;
    constexpr int V = IO<T>::V;
    constexpr int H = io2::H;
    constexpr int NWG = GT / 32;
    // rows of up to 4 packs per thread are widened to binary32 once and kept
    // in registers (unpacking them for each pass cost 50 % more instructions
    // at 16384 bf16); 8 packs per thread would not fit, so they are unpacked
    // again for each pass
    constexpr bool kWide = PACKS <= 4;
    static_assert(GT % 32 == 0 && (NWG & (NWG - 1)) == 0 && NWG >= 1 && NWG <= 32, "group size");
    static_assert(G >= 1 && G <= 15 && GT * G <= 1024, "groups per CTA");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float s1[G][2][NWG];
    __shared__ float2 s2[G][2][NWG];
    __shared__ __align__(8) uint64_t full[G][kMaxStages];
    __shared__ long long slot_row[G][kMaxStages];
    __shared__ unsigned long long next_row;

    const int g = threadIdx.x / GT;
    const int t = threadIdx.x % GT;
    const int bar_id = 1 + g;

    // balanced contiguous row range of this CTA
    const int64_t nb = gridDim.x, b = blockIdx.x;
    const int64_t q = a.rows / nb, rem = a.rows % nb;
    const int64_t r0 = b * q + (b < rem ? b : rem);
    const int64_t r1 = r0 + q + (b < rem ? 1 : 0);

    const int P = (int)(a.N / V);
    const uint32_t row_bytes = (uint32_t)(a.N * (int64_t)sizeof(T));
    const uint32_t stage_bytes = row_bytes * (OP == OP_ADD_RMS ? 2u : 1u);
    const int nparams = (OP == OP_LN) ? 2 : 1;
    const size_t params_bytes = smem_params == PARAMS_SMEM_F32 ? (size_t)nparams * (size_t)a.N * sizeof(float)
                                : smem_params == PARAMS_SMEM_RAW ? (size_t)nparams * (size_t)a.N * sizeof(T)
                                                                 : 0;
    unsigned char *ring = smem + params_bytes + (size_t)g * stages * stage_bytes;

#if NRM_ROW_PDL
    // programmatic dependent launch, as the other row kernels: the first rows
    // of the CTA's range are requested from L2 before the wait for the
    // previous grid (whose writes still reach the bulk copies issued after it)
    if (threadIdx.x == 0) {
        for (int64_t r = r0; r < r1 && r < r0 + (int64_t)G * stages; ++r) {
            prefetch_l2_bulk(static_cast<const T *>(a.x) + r * a.ldx, row_bytes);
            if (OP == OP_ADD_RMS) prefetch_l2_bulk(static_cast<const T *>(a.res) + r * a.ldr, row_bytes);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
#endif
    if (threadIdx.x == 0) next_row = (unsigned long long)r0;
    __syncthreads();
    int64_t issued = 0;  // leader: local row indices claimed so far
    int claim_s = 0;     // leader: the stage of the next claim (issued % stages)
    if (t == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[g][s], 1);
        fence_mbar_init();
        for (; issued < stages; ++issued)
            pipe_claim<OP, T>(a, &next_row, r1, slot_row[g], full[g], ring, stage_bytes, row_bytes,
                              (int)issued);
    }
    if (smem_params == PARAMS_SMEM_F32)
        fill_smem_params<T, (OP == OP_LN ? 2 : 1), GT * G>(a, reinterpret_cast<float *>(smem));
    else if (smem_params == PARAMS_SMEM_RAW)
        fill_smem_raw_params<T, (OP == OP_LN ? 2 : 1), GT * G>(a, reinterpret_cast<uint4 *>(smem));
    __syncthreads();

    const float fN = a.fN;
    const float invN = a.invN;
    const SmemParams<T> sprm{reinterpret_cast<const float4 *>(smem), P};
    const SmemRawParams<T> rprm{reinterpret_cast<const uint4 *>(smem), P, a.p0 != nullptr,
                                a.p1 != nullptr};
    const GlobalParams<T> gprm{static_cast<const T *>(a.p0), static_cast<const T *>(a.p1)};

    // row li of the group sits in stage s, whose phase parity is ph (kept
    // incrementally: a 64-bit division per row cost more than the row's
    // arithmetic)
    int64_t li = 0;
    int s = 0;
    uint32_t ph = 0;
    bool gave_up = false;
    for (;; ++li, s = s + 1 == stages ? 0 : s + 1, ph ^= (s == 0)) {
        const int par = (int)(li & 1);
        const bool ok = mbar_wait_bounded(&full[g][s], ph, a.wait_limit);
        if (!ok) atomicOr(a.fault, FAULT_WAIT);
        const int64_t row = slot_row[g][s];
        const bool valid = ok && row >= 0;
        const uint4 *st = reinterpret_cast<const uint4 *>(ring + (size_t)s * stage_bytes);

        // the row's raw packs (add+RMS: the rounded residual-stream packs,
        // also stored as residual_out); with kWide also widened once
        uint4 raw[PACKS];
        float2 v[kWide ? PACKS : 1][H];
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            const int idx = t + k * GT;
            if (idx < P) {
                raw[k] = st[idx];
                if (OP == OP_ADD_RMS) {
                    const uint4 rr = st[P + idx];
                    float2 fx[H], fr[H];
                    io2::unpack(raw[k], fx);
                    io2::unpack(rr, fr);
#pragma unroll
                    for (int h = 0; h < H; ++h) fx[h] = __fadd2_rn(fx[h], fr[h]);
                    raw[k] = io2::pack(fx);  // round once to T
                    if (valid)
                        st_stream(static_cast<T *>(a.res_out) + row * a.ldro + (size_t)idx * V, raw[k]);
                }
                if constexpr (kWide) io2::unpack(raw[k], v[k]);
            } else if constexpr (kWide) {
#pragma unroll
                for (int h = 0; h < H; ++h) v[k][h] = f2(0.f);  // contributes nothing
            }
        }
        // the values of pack k (kWide: the registers; else unpacked again)
        auto vals = [&](int k, float2 *f) {
            if constexpr (kWide) {
#pragma unroll
                for (int h = 0; h < H; ++h) f[h] = v[k][h];
            } else {
                io2::unpack(raw[k], f);
            }
        };

        // pass 1: sum (LayerNorm) or sum of squares (RMS ops)
        float2 acc = f2(0.f);
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            if (kWide || t + k * GT < P) {
                float2 f[H];
                vals(k, f);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    acc = (OP == OP_LN) ? __fadd2_rn(acc, f[h]) : __ffma2_rn(f[h], f[h], acc);
            }
        }
        bool stop;
        const float tot = group_cta_sum_or<NWG>(acc.x + acc.y, &s1[g][par][0], bar_id, !valid, stop);
        if (stop) {
            // A clean end is a completed phase carrying the sentinel; anything
            // else means some thread of the group gave up waiting.
            gave_up = !(ok && row < 0);
            break;  // the whole group leaves here together
        }
        if (t == 0 && issued < li + stages + 1) {
            // every thread holds this row in registers: refill its stage
            fence_proxy_async_smem();
            pipe_claim<OP, T>(a, &next_row, r1, slot_row[g], full[g], ring, stage_bytes, row_bytes,
                              claim_s);
            ++issued;
            claim_s = claim_s + 1 == stages ? 0 : claim_s + 1;
        }

        float rstd, m0 = 0.f, c = 0.f;
        if (OP == OP_LN) {
            // m0 = tot / N, corrected once so a constant row gives m0 == x
            m0 = tot * invN;
            m0 = fmaf(fmaf(-m0, fN, tot), invN, m0);
            const float2 nm = f2(-m0);
            float2 e1 = f2(0.f), e2 = f2(0.f);
#pragma unroll
            for (int k = 0; k < PACKS; ++k) {
                if (t + k * GT < P) {
                    float2 f[H];
                    vals(k, f);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 e = __fadd2_rn(f[h], nm);
                        if constexpr (kWide) v[k][h] = e;
                        e1 = __fadd2_rn(e1, e);
                        e2 = __ffma2_rn(e, e, e2);
                    }
                }
            }
            const float2 E = group_cta_sum<NWG>(make_float2(e1.x + e1.y, e2.x + e2.y),
                                                &s2[g][par][0], bar_id);
            c = E.x * invN;
            const float var = fmaxf(fmaf(-c, c, E.y * invN), 0.f);
            rstd = rsqrtf(var + a.eps);
            if (t == 0) {
                if (a.mean) a.mean[row] = m0 + c;
                if (a.rstd) a.rstd[row] = rstd;
            }
        } else {
            rstd = rsqrtf(fmaf(tot, invN, a.eps));
            if (t == 0 && a.rstd) a.rstd[row] = rstd;
        }

        // pass 3: normalize, scale (and shift), round once, store; LayerNorm
        // computes ((x - m0) - c) * rstd * gamma + beta either way
        T *Y = static_cast<T *>(a.y) + row * a.ldy;
        const float2 r2 = f2(rstd), nm = f2(kWide ? 0.f : -m0), nc = f2(-c);
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            const int idx = t + k * GT;
            if (idx < P) {
                float2 f[H], g2[H], out[H];
                vals(k, f);
                if (smem_params == PARAMS_SMEM_RAW) rprm.p0_pack(idx, g2);
                else if (smem_params) sprm.p0_pack(idx, g2);
                else gprm.p0_pack(idx, g2);
                if (OP == OP_LN) {
                    float2 b2[H];
                    if (smem_params == PARAMS_SMEM_RAW) rprm.p1_pack(idx, b2);
                    else if (smem_params) sprm.p1_pack(idx, b2);
                    else gprm.p1_pack(idx, b2);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 e = kWide ? f[h] : __fadd2_rn(f[h], nm);
                        out[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(e, nc), r2), g2[h], b2[h]);
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < H; ++h) out[h] = __fmul2_rn(__fmul2_rn(f[h], r2), g2[h]);
                }
                st_stream(Y + (size_t)idx * V, io2::pack(out));
            }
        }
    }

    // After a give-up: wait (bounded) for this group's copies still in flight,
    // the latest claimed index of each stage from li on, before exiting.
    if (t == 0 && gave_up) {
        for (int s = 0; s < stages; ++s) {
            int64_t j = -1;
            for (int64_t k = issued - 1; k >= li && k >= issued - stages; --k)
                if (k % stages == s) { j = k; break; }
            if (j >= 0 && slot_row[g][s] >= 0 &&
                !mbar_wait_bounded(&full[g][s], (uint32_t)((j / stages) & 1), 1u << 22))
                atomicOr(a.fault, FAULT_DRAIN);
        }
    }
}
