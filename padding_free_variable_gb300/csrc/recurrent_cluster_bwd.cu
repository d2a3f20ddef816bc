// recurrent_cluster_bwd.cu -- BPTT of the cluster-resident recurrent kernels and the db /
// dpeep sums (the forward kernels and the design notes are in recurrent_cluster.cu).
#include "recurrent_cluster.cuh"

namespace lstm {

// ------------------------------------------------------------------------- backward
//
// BPTT of the same recurrence ("Single Stream Parallelization...", Sec. 2) in
// the same cluster layout.  The error reaching h_t through R is
// R^T da_{t+1}; CTA c holds its 128 gate rows of R (as R^T, in tensor memory)
// and the gate errors it computes for them, so it forms the partial product
// P_c = R_c^T da_c for every unit on the tensor cores, and sends the part of
// P_c that belongs to CTA c' (its 32 units) into c''s inbox.  At the next step
// each CTA adds the G partials of its units in CTA order.  db and dpeep are
// summed afterwards by lstm_param_sums_kernel.
// Shared memory (RecArgs offsets): off_contrib = B (gate errors, NP pieces),
// off_acc = inbox, off_state = dc carry, off_sums = mbarriers, TMEM slot,
// failure flag, the group's step count, off_peep = peepholes, off_tab =
// tables; BULK also off_h = staging of the outgoing partials [G][NBM][32];
// with a.tma_pre off_red = operand tiles [7][NBM][32] (gates i f z o, c_t,
// c_{t-1}, dy).  Tensor memory: accumulators (tile m, chain ch) at columns
// (m * chains + ch) * NBM; piece k of R^T tile m from column
// tm_acol + 64 MT k + 64 m.  Sequence groups as in the forward kernel.
//
// Exchanges of the partials:
//  * BULK: the inbox is double-buffered per step parity ([2][G][NBM][32]);
//    the TMEM read-out lands in a staging buffer laid out per owner, and one
//    cp.async.bulk per owner copies it into the owner's inbox, completing on
//    the owner's mbarrier of that parity (re-armed before the CTA's own copies
//    go out, as in the forward kernel).  Warp w reads out owners w and w + 8
//    and issues their copies itself, each right after its own stores, so no
//    CTA barrier delays a copy.  A source can only write parity
//    (s & 1) again for step s + 2 after it received this CTA's partials of
//    step s + 1, which are formed after this CTA's cell of step s has read the
//    inbox.
// The cell's own operands arrive as TMA tiles when they fit (a.tma_pre),
// issued after the barrier that follows the cell (every thread has read them).
//  * otherwise: one inbox written with plain DSMEM stores between the two
//    halves of a split cluster barrier.
template <int NP, bool BULK, int U>
__global__ void __launch_bounds__(kCT, 1) lstm_rec_bwd_cluster_kernel(RecArgs a,
                                                                     const __grid_constant__ CUtensorMap map_ga,
                                                                     const __grid_constant__ CUtensorMap map_c,
                                                                     const __grid_constant__ CUtensorMap map_dy)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    cg::cluster_group cl = cg::this_cluster();
    const int G = a.G;
    const int rank = (int)cl.block_rank();
    const int ng = a.ngroups;
    const int dir = (int)(blockIdx.x / G) / ng, grp = (int)(blockIdx.x / G) % ng;
    const int S = a.grp_rows, j0 = grp * S;           // this cluster's sorted slots [j0, j0 + S)
    const int srank = grp == 0 ? rank : -1;           // the phase stamps come from group 0
    const int H = a.H, T = a.T, NBM = a.JC;
    const int MT = (H + kCM - 1) / kCM;              // 128-unit tiles of the partial product
    const int u0 = rank * kCU;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    const int nch = a.tm_chains;                     // chains per tile; issuers = MT * nch
    uint8_t* Bb = base + a.off_contrib;              // [NP][2 k-blocks][NBM][128 B]
    const size_t bsz = (size_t)2 * NBM * 128;        // bytes of one B piece
    float* inbox = reinterpret_cast<float*>(base + a.off_acc);       // [BULK ? 2 : 1][G][NBM][32]
    float* stage = reinterpret_cast<float*>(base + a.off_h);         // BULK: [G][NBM][32]
    float* tiles = reinterpret_cast<float*>(base + a.off_red);       // BULK + tma_pre: [7][NBM][32]
    float* dcc = reinterpret_cast<float*>(base + a.off_state);       // [S][32]
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(base + a.off_sums);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
    int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);
    uint64_t* full_bar = mma_bar + 2;                                // BULK: [2] inbox arrival per parity
    uint64_t* opnd_bar = mma_bar + 4;                                // operand tiles' arrival
    int* s_tg = reinterpret_cast<int*>(mma_bar + 6);                 // the group's step count
    float* peep_s = reinterpret_cast<float*>(base + a.off_peep);
    int* s_bs = reinterpret_cast<int*>(base + a.off_tab);            // [T] the group's active rows
    int* s_off = s_bs + T;                                           // [T+1] the group's first row
    int* s_len = s_off + T + 1;                                      // [S] lengths of the group's slots
    const uint32_t tcols = (uint32_t)a.Umax;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool tma_opnd = a.tma_pre != 0;
    auto inbox_at = [&](int parity, int src, int j) -> float* {
        return inbox + (((size_t)(BULK ? parity : 0) * G + src) * NBM + j) * kCU;
    };
    auto tile = [&](int k, int j) -> float* { return tiles + ((size_t)k * NBM + j) * kCU; };
    int Tg = 0;
    // rows of the partials of step s2 - 1 that step s2 reads: its rows with a step after them
    // (in recurrence order); the cell reads no others
    auto step_rows = [&](int s2) -> int {
        const int tp = dir == 0 ? Tg - s2 : s2 - 1, tn = dir == 0 ? Tg - 1 - s2 : s2;
        return min(s_bs[tp], s_bs[tn]);
    };
    // bytes a CTA receives for step s2: those rows from every other CTA (its own it writes itself)
    auto step_bytes = [&](int s2) -> uint32_t {
        return (uint32_t)(G - 1) * (uint32_t)step_rows(s2) * (uint32_t)(kCU * 4);
    };

    for (int i = threadIdx.x; i < NP * bsz / 16; i += kCT) reinterpret_cast<uint4*>(Bb)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < (BULK ? 2 : 1) * G * NBM * kCU; i += kCT) inbox[i] = 0.f;
    if (threadIdx.x == 0) *s_tg = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < T; i += kCT) {
        const int n = min(max(a.bs[i] - j0, 0), S);
        s_bs[i] = n;
        if (n > 0 && (i + 1 == T || a.bs[i + 1] <= j0)) *s_tg = i + 1;
    }
    for (int i = threadIdx.x; i <= T; i += kCT) s_off[i] = a.off[i] + j0;
    for (int i = threadIdx.x; i < S; i += kCT) s_len[i] = j0 + i < a.B ? a.slot_len[j0 + i] : 0;
    for (int i = threadIdx.x; i < 3 * kCU; i += kCT) {
        const int q = i / kCU, uu = i - q * kCU;
        peep_s[i] = a.peep[(size_t)dir * 3 * H + q * H + u0 + uu];
    }
    __syncthreads();
    Tg = *s_tg;
    if (threadIdx.x == 0) {
        tc::mbar_init(mma_bar, (uint32_t)(MT * nch));
        *s_fail = 0;
        if (BULK) {
            tc::mbar_init(&full_bar[0], 1);
            tc::mbar_init(&full_bar[1], 1);
        }
        if (tma_opnd) tc::mbar_init(opnd_bar, 1);
        tc::fence_mbar_init();
        // the inbox of step 1 (parity 1) is armed before the cluster barrier below
        if (BULK && Tg > 1) tc::mbar_arrive_expect_tx(&full_bar[1], step_bytes(1));
    }
    if (threadIdx.x < 32) {
        tc::tmem_alloc(tmem_slot, tcols);
        tc::tmem_relinquish();
    }
    fence_proxy_async_cta();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a0 = tmem + (uint32_t)a.tm_acol, ap = (uint32_t)(64 * MT);
    // R^T slice -> tensor memory: tile m, lane l = unit 128m + l (zero past H); column 64m + c
    // holds this CTA's gate rows r = 2c, 2c + 1 (r = 32g + uu); warps q and q + 4 share the
    // lanes 32q.. and take alternate gates
    {
        const int q = warp & 3;
        const uint32_t lanes = (uint32_t)(32 * q) << 16;
        for (int m = 0; m < MT; ++m) {
            const int up = 128 * m + 32 * q + lane;
            for (int g = warp >> 2; g < 4; g += 2) {
                float v[32];
#pragma unroll
                for (int uu = 0; uu < 32; ++uu) {
                    const size_t src = (size_t)dir * 4 * H * H + (size_t)(g * H + u0 + uu) * H + up;
                    v[uu] = up < H ? (NP > 1 ? __ldg(reinterpret_cast<const float*>(a.R) + src)
                                             : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.R)[src]))
                                   : 0.f;
                }
                uint32_t pc[NP][16];
                split32<NP>(v, pc);
#pragma unroll
                for (int k = 0; k < NP; ++k)
                    tc::tmem_st_32x32b_x16(a0 + (uint32_t)k * ap + lanes + (uint32_t)(64 * m + 16 * g), pc[k]);
            }
        }
        tc::tmem_wait_st();
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    // tma_opnd: the seven operand tiles of step s2 (NBM rows each; rows past the packed rows read
    // 0), one thread, completing on opnd_bar
    auto issue_opnd = [&](int s2) {
        const int t2 = dir == 0 ? Tg - 1 - s2 : s2;
        const int y0 = s_off[t2];
        const int yp = dir == 0 ? (t2 >= 1 ? s_off[t2 - 1] : 0) : (t2 + 1 < Tg ? s_off[t2 + 1] : 0);
        tc::mbar_arrive_expect_tx(opnd_bar, (uint32_t)(7 * NBM * kCU * 4));
#pragma unroll
        for (int g = 0; g < 4; ++g) tc::tma_load_2d(tile(g, 0), &map_ga, opnd_bar, dir * 4 * H + g * H + u0, y0);
        tc::tma_load_2d(tile(4, 0), &map_c, opnd_bar, dir * H + u0, y0);
        tc::tma_load_2d(tile(5, 0), &map_c, opnd_bar, dir * H + u0, yp);
        tc::tma_load_2d(tile(6, 0), &map_dy, opnd_bar, dir * H + u0, y0);
    };
    int last_tile = -1;                   // tile issuer: the last step whose tiles were issued
    if (tma_opnd && threadIdx.x == kTileIssuer && Tg > 0) { issue_opnd(0); last_tile = 0; }
    cl.sync();

    // cell item: row jq (+ RPP k), units uq .. uq + U: U units a thread, 32 / U threads a row
    constexpr int CPR = 32 / U, RPP = kCT / CPR;
    const int jq = threadIdx.x / CPR, qc = threadIdx.x % CPR, uq = qc * U;
    using PkT = typename PkU<U>::T;
    const uint32_t bstep = (uint32_t)(NBM * 128) >> 4;
    float pk[3][U];                                                  // peepholes i, f, o of units uq .. + U
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
        for (int e = 0; e < U; ++e) pk[q][e] = peep_s[q * kCU + uq + e];
    // c0 of slot j's units u0 + uq .. + U (the state before its first step; zero without one)
    auto init_c = [&](int j, float (&v)[U]) {
        if (a.c0) {
            ldg_u<U>(a.c0 + ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + uq, v);
        } else {
#pragma unroll
            for (int e = 0; e < U; ++e) v[e] = 0.f;
        }
    };
    // own operands (gates, c_t, c_{t-1}, dy) of row jq of a step, loaded one step ahead
    // (without operand tiles)
    float nx[7][U];
    auto load_own = [&](int s2) {
        const int t2 = dir == 0 ? Tg - 1 - s2 : s2;
        const int n2 = s_bs[t2];
        if (jq >= n2) return;
        const int row = s_off[t2] + jq;
        const float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + uq;
#pragma unroll
        for (int g = 0; g < 4; ++g) ld_u<U>(gr + g * H, nx[g]);
        const size_t yo = (size_t)row * ndH + dir * H + u0 + uq;
        ldg_u<U>(a.cbuf + yo, nx[4]);
        ldg_u<U>(a.dy + yo, nx[6]);
        const int np2 = dir == 0 ? (t2 >= 1 ? n2 : 0) : (t2 + 1 < Tg ? s_bs[t2 + 1] : 0);
        if (jq < np2) {
            const int pb2 = dir == 0 ? s_off[t2 - 1] : s_off[t2 + 1];
            ldg_u<U>(a.cbuf + (size_t)(pb2 + jq) * ndH + dir * H + u0 + uq, nx[5]);
        } else {
            init_c(jq, nx[5]);
        }
    };
    if (!tma_opnd && Tg > 0) load_own(0);
    bool failed = false;                  // CTA-uniform: a bounded wait ran out
    bool step_ok = true;                  // this thread's wait of the last product
    for (int s = 0; s < Tg; ++s) {
        const int t = dir == 0 ? Tg - 1 - s : s;
        const int n = s_bs[t];
        const int rowbase = s_off[t];
        const int n_next = dir == 0 ? (t + 1 < Tg ? s_bs[t + 1] : 0) : (t >= 1 ? n : 0);
        const int prev_base = dir == 0 ? (t >= 1 ? s_off[t - 1] : 0) : (t + 1 < Tg ? s_off[t + 1] : 0);
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < Tg ? s_bs[t + 1] : 0);
        const int NBs = (n + 15) & ~15;
        const int par = BULK ? (s & 1) : 0;
        cstamp(a, true, dir, srank, s, 0, 0);
        bool arrived = true;              // this step's inbox and operand tiles arrived
        if (BULK && s > 0 && !failed)
            arrived = tc::mbar_wait(&full_bar[par], (uint32_t)(((s - 1) >> 1) & 1), a.wait_limit_ns);
        if (tma_opnd && !failed && !tc::mbar_wait(opnd_bar, (uint32_t)(s & 1), a.wait_limit_ns)) arrived = false;
        if (!arrived && !failed) {
            record_failure(a.status, LSTM_ERR_TIMEOUT, 0x60000u | (unsigned)s);
            *s_fail = 1 + s;
        }
        cstamp(a, true, dir, srank, s, 1, 1);
        for (int it = 0; it * RPP < n; ++it) {
            const int j = jq + it * RPP;
            if (j >= n) continue;
            const int row = rowbase + j;
            float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + uq;
            float gv[4][U], cv[U], cpv[U], dyv[U];
            if (tma_opnd) {
#pragma unroll
                for (int g = 0; g < 4; ++g) ld_u<U>(tile(g, j) + uq, gv[g]);
                ld_u<U>(tile(4, j) + uq, cv);
                ld_u<U>(tile(6, j) + uq, dyv);
                if (j < n_prev) ld_u<U>(tile(5, j) + uq, cpv);
                else init_c(j, cpv);
            } else if (it == 0) {
#pragma unroll
                for (int e = 0; e < U; ++e) {
                    gv[0][e] = nx[0][e]; gv[1][e] = nx[1][e]; gv[2][e] = nx[2][e]; gv[3][e] = nx[3][e];
                    cv[e] = nx[4][e]; cpv[e] = nx[5][e]; dyv[e] = nx[6][e];
                }
            } else {
#pragma unroll
                for (int g = 0; g < 4; ++g) ld_u<U>(gr + g * H, gv[g]);
                const size_t yo = (size_t)row * ndH + dir * H + u0 + uq;
                ldg_u<U>(a.cbuf + yo, cv);
                ldg_u<U>(a.dy + yo, dyv);
                if (j < n_prev) ldg_u<U>(a.cbuf + (size_t)(prev_base + j) * ndH + dir * H + u0 + uq, cpv);
                else init_c(j, cpv);
            }
            const bool has_next = j < n_next;
            const bool real = !a.padded || t < s_len[j];
            // the G partial sums of R^T da of the step after, added in CTA order, and the carry
            float dhr[U], car[U];
#pragma unroll
            for (int e = 0; e < U; ++e) { dhr[e] = 0.f; car[e] = 0.f; }
            const size_t so = ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + uq;   // caller-order state
            if (has_next) {
                for (int c2 = 0; c2 < G; ++c2) {
                    float x[U];
                    ld_u<U>(inbox_at(par, c2, j) + uq, x);
#pragma unroll
                    for (int e = 0; e < U; ++e) dhr[e] += x[e];
                }
                ld_u<U>(dcc + j * kCU + uq, car);
            } else {
                // the sequence's last step: the final state's own errors from outside
                if (a.dh_n) ldg_u<U>(a.dh_n + so, dhr);
                if (a.dc_n) ldg_u<U>(a.dc_n + so, car);
            }
            float da[4][U], cout[U];
#pragma unroll
            for (int e = 0; e < U; ++e) {
                float dai = 0.f, daf = 0.f, daz = 0.f, dao = 0.f, carry_out = 0.f;
                if (real) {
                    const float ig = gv[0][e], fg = gv[1][e], zg = gv[2][e], og = gv[3][e];
                    const float c = cv[e], cp = cpv[e];
                    const float dh = dyv[e] + dhr[e];
                    const float tc = tanh_c(c);
                    dao = dh * tc * og * (1.f - og);
                    const float dc = dh * og * (1.f - tc * tc) + dao * pk[2][e] + car[e];
                    dai = dc * zg * ig * (1.f - ig);
                    daf = dc * cp * fg * (1.f - fg);
                    daz = dc * ig * (1.f - zg * zg);
                    carry_out = dc * fg + dai * pk[0][e] + daf * pk[1][e];
                }
                da[0][e] = dai; da[1][e] = daf; da[2][e] = daz; da[3][e] = dao;
                cout[e] = carry_out;
            }
            st_u<U>(dcc + j * kCU + uq, cout);
            if (j >= n_prev && a.dc0) st_u<U>(a.dc0 + so, cout);   // the sequence's first step: dL/dc0
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                st_u<U>(gr + g * H, da[g]);
                PkT pc[NP];
                split_u<U, NP>(da[g], pc);
                const uint32_t o = sw_off4(j, g * kCU + uq, NBM);
#pragma unroll
                for (int k = 0; k < NP; ++k) *reinterpret_cast<PkT*>(Bb + (size_t)k * bsz + o) = pc[k];
            }
        }
        if (BULK) cstamp(a, true, dir, srank, s, 4, 4);   // (BULK: stamp 4 = cell done)
        if (!BULK) cluster_arrive_relaxed();   // this CTA has read its inbox: peers may overwrite it
        // the previous step's staging must have been read by its copies before this step's read-out
        if (BULK && lane == 0 && warp < G) bulk_wait_read_all();
        fence_proxy_async_cta();
        // a timeout (of the previous step's product, or of this step's arrivals) becomes a
        // CTA-uniform decision here, before the next issue: from then on the CTA issues, waits
        // for, re-arms and sends nothing (that step's read-out may have seen partial sums; the
        // status word marks the results as invalid)
        if (__syncthreads_or(!step_ok || !arrived)) failed = true;
        // the operand tiles and this parity's inbox have been read
        if (tma_opnd && threadIdx.x == kTileIssuer && s + 1 < Tg && !failed) {
            issue_opnd(s + 1);
            last_tile = s + 1;
        }
        // BULK: re-arm this parity for step s + 2 before this CTA's partials of step s go out
        if (BULK && threadIdx.x == 0 && !failed && s + 2 < Tg)
            tc::mbar_arrive_expect_tx(&full_bar[par], step_bytes(s + 2));
        cstamp(a, true, dir, srank, s, 2, 2);
        if (s + 1 < Tg) {
            // P[u'][j] = sum over this CTA's gate rows r of R[r][u'] da[j][r]: warp w issues tile
            // m = w / chains, chain ch = w % chains (k-steps ch, ch + chains, ... of the 8)
            if (lane == 0 && warp < MT * nch && !failed) {
                tc::tc_fence_after_sync();
                const int m = warp / nch, ch = warp - m * nch;
                const uint32_t idesc = tc::idesc_bf16_f32(kCM, NBs);
                const uint64_t db0 = tc::sdesc_sw128(tc::smem_u32(Bb)), bp = (uint64_t)(bsz >> 4);
                const uint32_t dm = tmem + (uint32_t)(warp * NBM), am = a0 + (uint32_t)(64 * m);
                if (nch == 4) issue_chain_fixed<4, 8, 4, NP>(dm, am, ap, db0, bp, bstep, ch, idesc);
                else if (nch == 2) issue_chain_fixed<2, 8, 4, NP>(dm, am, ap, db0, bp, bstep, ch, idesc);
                else issue_chain_fixed<1, 8, 4, NP>(dm, am, ap, db0, bp, bstep, ch, idesc);
                if (!(s == 0 && dir == 0 && grp == 0 && rank == a.debug_skip_cta)) tc::mma_commit(mma_bar);   // test hook
            }
            if (warp < MT * nch) __syncwarp();
            cstamp(a, true, dir, srank, s, 6, 6);
            step_ok = failed ? true : tc::mbar_wait(mma_bar, (uint32_t)(s & 1), a.wait_limit_ns);
            if (!step_ok) {
                record_failure(a.status, LSTM_ERR_TIMEOUT, 0x50000u | (unsigned)s);
                *s_fail = 1 + s;
            }
            tc::tc_fence_after_sync();
            cstamp(a, true, dir, srank, s, 5, 7);
        }
        if (BULK) {
            if (s + 1 < Tg && !failed) {
                // read-out into the staging, per owner: tile m, lane quarter q -> owner 4m + q,
                // units 32q + lane of the tile, rows [0, NBs).  The warp that wrote an owner's
                // partial copies it to that owner at once (lane 0; warp w serves owners w, w + 8),
                // so no CTA barrier stands between a partial and its copy
                const uint32_t nxt = (uint32_t)(par ^ 1);
                const uint32_t bytes = (uint32_t)step_rows(s + 1) * (uint32_t)(kCU * 4);
                // this CTA's own units go straight into its next inbox
                auto dst_of = [&](int owner) -> float* {
                    return owner == (int)rank ? inbox_at(par ^ 1, rank, 0) : stage + (size_t)owner * NBM * kCU;
                };
                auto send = [&](int owner) {
                    if (owner != (int)rank && bytes != 0) {
                        fence_proxy_async_cta();      // this lane's stores, visible to the copy
                        __syncwarp();
                        if (lane == 0)
                            bulk_to_peer(mapa_u32(tc::smem_u32(inbox_at(nxt, rank, 0)), (uint32_t)owner),
                                         stage + (size_t)owner * NBM * kCU, bytes,
                                         mapa_u32(tc::smem_u32(&full_bar[nxt]), (uint32_t)owner));
                    }
                };
                const int o0 = warp, o1 = warp + kCT / 32;     // at most two owners a warp
                const bool h0 = o0 < MT * 4 && o0 < G, h1 = o1 < MT * 4 && o1 < G;
                if (NBs == 16 && MT * 4 <= 2 * (kCT / 32) && ((int)h0 + (int)h1) * nch <= 2) {
                    // one column block and at most two accumulator loads a warp (two owners of one
                    // chain, or one owner of two chains): all loads in flight together
                    const uint32_t t0 = tmem + ((uint32_t)((o0 & 3) * 32) << 16) + (uint32_t)((o0 >> 2) * nch * NBM);
                    const uint32_t t1 = tmem + ((uint32_t)((o1 & 3) * 32) << 16) + (uint32_t)((o1 >> 2) * nch * NBM);
                    uint32_t r0[16], r1[16];
                    if (h0) tc::tmem_ld_32x32b_x16(t0, r0);
                    if (h1) tc::tmem_ld_32x32b_x16(t1, r1);
                    else if (h0 && nch == 2) tc::tmem_ld_32x32b_x16(t0 + (uint32_t)NBM, r1);   // o0's second chain
                    tc::tmem_wait_ld();
                    if (h0) {
                        float* dst = dst_of(o0);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float v = __uint_as_float(r0[e]);
                            if (nch == 2) v += __uint_as_float(r1[e]);
                            dst[(size_t)e * kCU + lane] = v;
                        }
                        send(o0);
                    }
                    if (h1) {
                        float* dst = dst_of(o1);
#pragma unroll
                        for (int e = 0; e < 16; ++e) dst[(size_t)e * kCU + lane] = __uint_as_float(r1[e]);
                        send(o1);
                    }
                } else {
                    for (int pq = warp; pq < MT * 4; pq += kCT / 32) {
                        const int m = pq >> 2, q = pq & 3;
                        const int owner = 4 * m + q;
                        if (owner >= G) continue;
                        float* dst = dst_of(owner);
                        for (int c0 = 0; c0 < NBs; c0 += 16) {
                            float v[16];
                            tmem_sum_chains(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * nch * NBM + c0),
                                            (uint32_t)NBM, nch, v);
#pragma unroll
                            for (int e = 0; e < 16; ++e) dst[(size_t)(c0 + e) * kCU + lane] = v[e];
                        }
                        send(owner);
                    }
                }
                if (lane == 0 && warp < G) bulk_commit();
            }
            tc::tc_fence_before_sync();
            __syncthreads();      // this CTA's own partial (in its next inbox) is visible to every thread
            if (!tma_opnd && s + 1 < Tg) load_own(s + 1);   // the next step's own operands
            cstamp(a, true, dir, srank, s, 3, 3);
        } else {
            cluster_wait();        // every peer has read its inbox of this step
            if (s + 1 < Tg && !failed) {
                // tile m, lane quarter q: units u' = 128m + 32q + lane, owned by CTA 4m + q
                for (int pq = warp; pq < MT * 4; pq += kCT / 32) {
                    const int m = pq >> 2, q = pq & 3;
                    const int owner = 4 * m + q;
                    if (owner >= G) continue;
                    float* dst_base = cl.map_shared_rank(inbox_at(0, rank, 0), owner);
                    for (int c0 = 0; c0 < NBs; c0 += 16) {
                        float v[16];
                        tmem_sum_chains(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * nch * NBM + c0),
                                        (uint32_t)NBM, nch, v);
                        // lanes are consecutive units: each store is one coalesced 128-byte row
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + e < n) dst_base[(size_t)(c0 + e) * kCU + lane] = v[e];
                    }
                }
                tc::tc_fence_before_sync();
            }
            cstamp(a, true, dir, srank, s, 3, 3);
            fence_proxy_async_cluster();
            cluster_arrive();      // release: this CTA's partial sums are in their owners' inboxes
            if (!tma_opnd && s + 1 < Tg) load_own(s + 1);   // the next step's own operands, in flight across the barrier
            cluster_wait();
            cstamp(a, true, dir, srank, s, 4, 4);
        }
    }
    // after a timeout the last tiles issued may not have been waited for (bounded wait)
    if (tma_opnd && threadIdx.x == kTileIssuer && last_tile >= 0)
        tc::mbar_wait(opnd_bar, (uint32_t)(last_tile & 1), kTeardownWaitNs);
    if (BULK) {
        if (lane == 0 && warp < G) bulk_wait_all();   // no copy of this CTA is still in flight
        cl.sync();                                    // nor one into it
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        __syncwarp();
        tc::tc_fence_after_sync();
        if (failed) tc::mbar_wait(mma_bar, (uint32_t)((*s_fail - 1) & 1), kTeardownWaitNs);
        tc::tmem_dealloc(tmem, tcols);
    }
}

// db and dpeep from the gate errors: column (direction, quantity q, unit u),
// q = 0..3 -> sum of da_q, 4 -> da_i c_{t-1}, 5 -> da_f c_{t-1}, 6 -> da_o c_t.
// Thread (direction, unit) takes all seven columns of its unit over one chunk of
// rows, in row order, so each row's gate errors and states are read once; the
// chunks are then added in chunk order (bitwise repeatable).  c_{t-1} of a
// sequence's first step is its initial state c0 (zero when c0 is null).
__global__ void lstm_param_sums_kernel(const float* __restrict__ ga, const float* __restrict__ cbuf,
                                       const int32_t* __restrict__ prev_fwd, const int32_t* __restrict__ prev_rev,
                                       const float* __restrict__ c0, const int32_t* __restrict__ row_slot,
                                       const int32_t* __restrict__ perm, int B,
                                       int rows, int H, int ndir, int chunk, float* __restrict__ partial)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= ndir * H) return;
    const int d = t / H, u = t - d * H;
    const int r0 = blockIdx.y * chunk, r1 = min(rows, r0 + chunk);
    const int nd4H = ndir * 4 * H, ndH = ndir * H;
    const int32_t* prev = d == 0 ? prev_fwd : prev_rev;
    float s[7] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int r = r0; r < r1; ++r) {
        const float* g = ga + (size_t)r * nd4H + (size_t)d * 4 * H + u;
        const float ai = __ldg(g), af = __ldg(g + H), az = __ldg(g + 2 * H), ao = __ldg(g + 3 * H);
        const int pr = __ldg(prev + r);
        const float cp = pr >= 0 ? __ldg(cbuf + (size_t)pr * ndH + d * H + u)
                       : c0 ? __ldg(c0 + ((size_t)d * B + __ldg(perm + __ldg(row_slot + r))) * H + u) : 0.f;
        const float ct = __ldg(cbuf + (size_t)r * ndH + d * H + u);
        s[0] += ai; s[1] += af; s[2] += az; s[3] += ao;
        s[4] += ai * cp; s[5] += af * cp; s[6] += ao * ct;
    }
    float* out = partial + (size_t)blockIdx.y * ndir * 7 * H + (size_t)d * 7 * H + u;
#pragma unroll
    for (int q = 0; q < 7; ++q) out[(size_t)q * H] = s[q];
}

__global__ void lstm_param_sums_combine(const float* __restrict__ partial, int chunks, int H, int ndir,
                                        float* __restrict__ db, float* __restrict__ dpeep)
{
    const int ncols = ndir * 7 * H;
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= ncols) return;
    float s = 0.f;
    for (int c = 0; c < chunks; ++c) s += partial[(size_t)c * ncols + col];
    const int d = col / (7 * H), rem = col - d * 7 * H, q = rem / H, u = rem - q * H;
    if (q < 4) db[(size_t)d * 4 * H + q * H + u] = s;
    else dpeep[(size_t)d * 3 * H + (q - 4) * H + u] = s;
}

// ------------------------------------------------------------------------- configuration
template <int U>
static const void* bwd_kernel_u(bool bf16, bool bulk)
{
    if (bulk) return bf16 ? (const void*)lstm_rec_bwd_cluster_kernel<1, true, U>
                          : (const void*)lstm_rec_bwd_cluster_kernel<3, true, U>;
    return bf16 ? (const void*)lstm_rec_bwd_cluster_kernel<1, false, U> : (const void*)lstm_rec_bwd_cluster_kernel<3, false, U>;
}
static const void* bwd_kernel(bool bf16, bool bulk, int group_rows)
{
    return cell_units(group_rows, true) == 2 ? bwd_kernel_u<2>(bf16, bulk) : bwd_kernel_u<4>(bf16, bulk);
}

bool rec_cluster_bwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* lay)
{
    if (p.gemm_engine != 0 || p.forced_ctas != 0) return false;
    if (H % kCU != 0) return false;
    const int G = H / kCU;
    if (G > 16 || G * ndir > p.num_sms) return false;
    int S = 0, ng = 1;
    if (!choose_groups(p, G, ndir, &S, &ng)) return false;
    const int NBM = std::max(16, (std::min(S, max_active_rows(p)) + 15) & ~15);
    const int MT = (H + kCM - 1) / kCM;
    const int np = bf16 ? 1 : 3;                   // bf16 pieces of each operand
    const int acols = MT * 64 * np;                // R^T tiles in TMEM: 128 gate rows = 64 columns per piece
    int nch = 4;
    while (nch > 1 && (MT * nch > 4 || MT * nch * NBM + acols > 512)) nch >>= 1;
    if (MT * nch * NBM + acols > 512 || MT * nch > kCT / 32) return false;
    const uint32_t cols = pow2_cols(MT * nch * NBM + acols);
    // bulk exchange with operand tiles first, then the single-buffered barrier exchange with
    // and without tiles (the last needs the least shared memory)
    const int order[4][2] = {{1, 1}, {0, 1}, {0, 0}, {1, 0}};
    for (int oi = 0; oi < 4; ++oi) {
        const int bulk = order[oi][0], tiles = order[oi][1];
        if (oi == 3 && p.forced_variant < 0) break;   // the bulk exchange without tiles only on request
        if (p.forced_variant >= 0 && p.forced_variant != (bulk | tiles << 1)) continue;
        size_t off = 0;
        const size_t o_b = off; off = al(off + (size_t)np * 2 * NBM * 128, 1024);
        const size_t o_in = off; off = al(off + (bulk ? 2 : 1) * (size_t)G * NBM * kCU * 4, 1024);
        const size_t o_stage = off; if (bulk) off = al(off + (size_t)G * NBM * kCU * 4, 1024);
        const size_t o_tiles = off; if (tiles) off = al(off + 7 * (size_t)NBM * kCU * 4, 1024);
        const size_t o_dcc = off; off = al(off + (size_t)S * kCU * 4, 16);
        const size_t o_bar = off; off = al(off + 64, 16);
        const size_t o_peep = off; off = al(off + 3 * kCU * 4, 16);
        const size_t o_tab = off; off = al(off + (size_t)(2 * p.T + 1 + S) * 4, 16);
        size_t smem = off + 1024 + 64;
        smem = tmem_safe_smem(p, smem, cols);
        if (smem == 0) return false;
        if (!cluster_schedulable(p, bwd_kernel(bf16, bulk != 0, S), G, smem)) continue;
        RecConfig c;
        c.G = G; c.Umax = (int)cols; c.JC = NBM; c.smem = smem; c.cluster = 1;
        c.chains = nch; c.acol = (int)cols - acols; c.bulk = bulk; c.tma_pre = tiles;
        c.grp_rows = S; c.ngroups = ng;
        *out = c;
        lay->off_contrib = (int)o_b; lay->off_acc = (int)o_in; lay->off_h = (int)o_stage; lay->off_red = (int)o_tiles;
        lay->off_state = (int)o_dcc; lay->off_sums = (int)o_bar; lay->off_peep = (int)o_peep; lay->off_tab = (int)o_tab;
        return true;
    }
    return false;
}

size_t rec_cluster_bwd_sum_floats(int H, int ndir) { return (size_t)kSumChunks * ndir * 7 * H; }

lstm_status rec_cluster_bwd_launch(const Plan& p, const RecConfig& c, RecArgs a, float* sum_scratch, cudaStream_t s)
{
    a.G = c.G; a.Umax = c.Umax; a.JC = c.JC; a.tm_chains = c.chains; a.tm_acol = c.acol;
    a.grp_rows = c.grp_rows; a.ngroups = c.ngroups;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    const void* fn = bwd_kernel(a.bf16 != 0, c.bulk != 0, c.grp_rows);
    // operand tiles: ga as [rows][ndir*4H], c and dy as [rows][ndir*H] fp32, boxes of 32 x NBM
    CUtensorMap map_ga, map_c, map_dy;
    memset(&map_ga, 0, sizeof(map_ga));
    memset(&map_c, 0, sizeof(map_c));
    memset(&map_dy, 0, sizeof(map_dy));
    const int nd4H = a.ndir * 4 * a.H, ndH = a.ndir * a.H;
    a.tma_pre = c.tma_pre && make_map_f32(&map_ga, a.ga, p.rows, nd4H, nd4H, kCU, c.JC) &&
                make_map_f32(&map_c, a.cbuf, p.rows, ndH, ndH, kCU, c.JC) &&
                make_map_f32(&map_dy, a.dy, p.rows, ndH, ndH, kCU, c.JC) ? 1 : 0;
    void* args[] = {&a, &map_ga, &map_c, &map_dy};
    trace_begin(p, K_REC_BWD, s);
    lstm_status st = cluster_launch(c, fn, args, a.ndir, s);
    int launched = st == LSTM_OK ? 1 : 0;
    if (st == LSTM_OK) {
        st = param_sums_launch(p, a.ga, a.cbuf, a.H, a.ndir, a.db, a.dpeep, sum_scratch, s, a.c0);
        if (st == LSTM_OK) launched += 2;
    }
    trace_end(p, K_REC_BWD, s, launched);
    return st;
}

lstm_status param_sums_launch(const Plan& p, const float* ga, const float* cbuf, int H, int ndir, float* db,
                              float* dpeep, float* sum_scratch, cudaStream_t s, const float* c0)
{
    const int ncols = ndir * 7 * H;
    const int rows = (int)p.rows;
    const int chunk = (rows + kSumChunks - 1) / kSumChunks;
    lstm_param_sums_kernel<<<dim3((ndir * H + 127) / 128, kSumChunks), 128, 0, s>>>(
        ga, cbuf, p.d_prev_fwd, p.d_prev_rev, c0, p.d_row_slot, p.d_perm, p.B, rows, H, ndir, chunk, sum_scratch);
    lstm_param_sums_combine<<<(ncols + 255) / 256, 256, 0, s>>>(sum_scratch, kSumChunks, H, ndir, db, dpeep);
    return cudaGetLastError() == cudaSuccess ? LSTM_OK : LSTM_ERR_UNSUPPORTED;
}

}  // namespace lstm
