// recurrent_cluster.cu -- cluster-resident recurrent kernels (forward and BPTT).
//
// The same recurrence as lstm_rec_fwd_kernel ("Single Stream Parallelization
// of Generalized LSTM-Like RNNs on a GPU", Sec. 3: one sequential step per
// frame, the delayed connection R h_{t-1} then the cell), laid out for
// thread-block clusters when one direction's R fits in a cluster:
//
//  * sequence groups: the sorted slots are cut into contiguous groups of S
//    slots, and every (direction, group) pair is one cluster of G = H/32
//    CTAs.  Sequences are independent, so the clusters never communicate;
//    a group runs only as many steps as its longest sequence, and each
//    cluster moves only its own rows between its CTAs every step;
//  * CTA c of a cluster owns units [32c, 32c+32) and their 128 gate rows of
//    R, resident in TENSOR MEMORY as the MMA's A operand.  bf16 weights are
//    one bf16 piece; fp32 weights (and the fp32 B operands h_{t-1} or the
//    gate errors) are three bf16 pieces v0 + v1 + v2 (v0 = bf16(v), each
//    further piece the bf16 rounding of what the earlier ones leave), and
//    each K = 16 step issues the six piece products above 2^-24 of the
//    leading one, so the product keeps fp32 accuracy.  With A in tensor
//    memory an M=128, N<=32, K=16 MMA reads only its B tile from shared
//    memory (measured on GB300: ~19 cycles per MMA with 4 issuing warps,
//    against ~43 with A in shared memory);
//  * per step up to 4 warps each issue one chain of tcgen05.mma into their
//    own accumulator columns (chains summed at read-out); N is the group's
//    active rows rounded up to 16;
//  * the cell runs on the summed chains, and each CTA sends its h_t (bf16
//    pieces, swizzled) to every peer of its cluster.  Two exchanges:
//    BULK -- the operand is double-buffered per step parity; each CTA stages
//    its h_t and pushes it with one cp.async.bulk per peer and piece into the
//    peer's buffer of the other parity, completing on the peer's mbarrier of
//    that parity.  The data's arrival is the step's synchronisation: no
//    cluster barrier runs in the step loop.  Otherwise (the double buffers do
//    not fit): one operand buffer written with DSMEM stores between the two
//    halves of a split cluster barrier.
// Every wait but the hardware cluster barrier (which every CTA of a cluster
// reaches by construction) is bounded, and a timeout is recorded in the
// plan's status word.
#include "recurrent_cluster.cuh"

namespace lstm {

// Shared memory (RecArgs offsets): off_acc = accs, off_state = cell states,
// off_contrib = B operand (h_{t-1}, its NP pieces), off_sums = mbarriers, TMEM
// slot, failure flag and the group's step count, off_tab = tables, off_peep =
// peepholes.  Tensor memory: accumulator chains in columns [0, chains * NBM),
// the R slice (NP pieces of H/2 columns each) from column tm_acol.
//
// The cluster serves sorted slots [j0, j0 + S) of direction `dir`: its step t
// has rows off[t] + j0 .. + n - 1, n = min(max(bs[t] - j0, 0), S), and it runs
// the Tg steps with n > 0 (Tg = the group's longest length).
//
// Two exchanges of h_t between the CTAs of a cluster:
//  * BULK: the operand is double-buffered per step parity, in 32-unit blocks
//    of the 64-byte swizzled layout, so that one CTA's units of all rows are
//    one contiguous block.  Each CTA stages its h_t there in its own shared
//    memory and copies it with one cp.async.bulk per peer and piece, which
//    completes on the peer's mbarrier of that parity: the arrival of the
//    data is the step's synchronisation, and no cluster barrier runs inside
//    the step loop.  A peer can only send h_{t+1} into buffer (s & 1) after
//    it received this CTA's h_t, which is sent after this CTA's product of
//    step s has read that buffer; each mbarrier is re-armed for its next use
//    before this CTA's copies of the step go out, so no byte can arrive at an
//    unarmed barrier.
//  * otherwise (the double buffer does not fit): one operand buffer, written
//    by the peers with plain DSMEM stores between two halves of a split
//    cluster barrier.
//
// With a.tma_pre the gate pre-activations of a step (4 gates x NBM rows x this
// CTA's 32 units, fp32) arrive in shared memory by four TMA tile loads, issued
// by one thread right after the previous step's cell has read the tile: the
// product's window stays free of the 256 threads' global loads (measured to
// delay the MMAs' completion by ~0.8 us).
template <int NP, bool BULK, int U>
__global__ void __launch_bounds__(kCT, 1) lstm_rec_fwd_cluster_kernel(RecArgs a, const __grid_constant__ CUtensorMap pre_map)
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
    const int H = a.H, T = a.T, NBM = a.JC;          // JC carries the operand buffer rows (multiple of 16)
    const int KB = (H + 63) / 64;
    const int u0 = rank * kCU;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    const int nch = a.tm_chains;
    float* accs = reinterpret_cast<float*>(base + a.off_acc);        // [NBM][128]
    float* cst = reinterpret_cast<float*>(base + a.off_state);       // [S][32]
    // B operand: BULK [2 parity][NP][G][NBM][64 B], else [NP][KB][NBM][128 B]
    uint8_t* Bb = base + a.off_contrib;
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(base + a.off_sums);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
    int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);
    uint64_t* full_bar = mma_bar + 2;                                // BULK: [2] operand arrival per parity
    uint64_t* pre_bar = mma_bar + 4;                                 // tma_pre: arrival of a step's tile
    int* s_tg = reinterpret_cast<int*>(mma_bar + 6);                 // the group's step count
    float* pre_tile = reinterpret_cast<float*>(base + a.off_red);    // tma_pre: [4 gates][NBM][32]
    const bool tma_pre = a.tma_pre != 0;
    float* peep_s = reinterpret_cast<float*>(base + a.off_peep);     // [3][32]
    int* s_bs = reinterpret_cast<int*>(base + a.off_tab);            // [T] the group's active rows
    int* s_off = s_bs + T;                                           // [T+1] the group's first row
    int* s_len = s_off + T + 1;                                      // [S] lengths of the group's slots
    uint8_t* stage = base + a.off_h;                                 // BULK: [2 parity][NP][NBM][64 B]
    const size_t bsz = BULK ? (size_t)G * NBM * 64 : (size_t)KB * NBM * 128;   // bytes of one B piece
    const size_t ssz = (size_t)NBM * 64;                             // bytes of one staged h piece
    auto Bop = [&](int parity, int piece) -> uint8_t* {
        return Bb + (BULK ? (size_t)parity * NP * bsz : 0) + (size_t)piece * bsz;
    };
    auto Stg = [&](int parity, int piece) -> uint8_t* { return stage + (size_t)(parity * NP + piece) * ssz; };
    int Tg = 0;
    // rows of h of step s2 - 1 that step s2 reads: the rows continuing into step s2.  Rows past
    // them are never read going forward (finished sequences) and were never written going
    // backward (sequences not yet started: still zero from the set-up)
    auto step_rows = [&](int s2) -> int {
        const int tp = dir == 0 ? s2 - 1 : Tg - s2, tn = dir == 0 ? s2 : Tg - 1 - s2;
        return min(s_bs[tp], s_bs[tn]);
    };
    // bytes a CTA receives for step s2: those rows from every other CTA (its own it writes itself)
    auto step_bytes = [&](int s2) -> uint32_t {
        return (uint32_t)(G - 1) * (uint32_t)NP * (uint32_t)step_rows(s2) * 64u;
    };
    const uint32_t tcols = (uint32_t)a.Umax;                         // Umax carries the TMEM columns
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up: operand zeroed, the group's tables, barriers, tensor memory
    for (size_t i = threadIdx.x; i < (BULK ? 2 : 1) * NP * bsz / 16; i += kCT)
        reinterpret_cast<uint4*>(Bb)[i] = make_uint4(0, 0, 0, 0);
    if (BULK)
        for (size_t i = threadIdx.x; i < 2 * NP * ssz / 16; i += kCT) reinterpret_cast<uint4*>(stage)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) *s_tg = 0;
    __syncthreads();
    // bs is non-increasing in t, so the group's steps are t < Tg, Tg = the one t whose
    // successor has no row of the group
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
        tc::mbar_init(mma_bar, (uint32_t)nch);
        *s_fail = 0;
        if (BULK) {
            tc::mbar_init(&full_bar[0], 1);
            tc::mbar_init(&full_bar[1], 1);
        }
        if (tma_pre) tc::mbar_init(pre_bar, 1);
        tc::fence_mbar_init();
        // the operand of step 1 (parity 1) is armed before the cluster barrier below,
        // i.e. before any peer can send
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
    const uint32_t a0 = tmem + (uint32_t)a.tm_acol, ap = (uint32_t)(H / 2);
    // R slice -> tensor memory: lane 32g + uu holds gate row g of unit u0 + uu (the MMA's row
    // order), column c of the slice holds k = 2c and 2c + 1; warps g and g + 4 share the lanes
    // of gate g and take alternate 32-wide k chunks
    {
        const int g = warp & 3;
        const size_t grow = (size_t)dir * 4 * H * H + (size_t)(g * H + u0 + lane) * H;
        const uint32_t lanes = (uint32_t)(32 * g) << 16;
        for (int cc = warp >> 2; cc < H / 32; cc += 2) {
            float v[32];
            if (NP > 1) {
                const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.R) + grow + 32 * cc);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 x = __ldg(src + e);
                    v[4 * e] = x.x; v[4 * e + 1] = x.y; v[4 * e + 2] = x.z; v[4 * e + 3] = x.w;
                }
            } else {
                const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(a.R) + grow + 32 * cc;
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __bfloat162float(src[e]);
            }
            uint32_t pc[NP][16];
            split32<NP>(v, pc);
#pragma unroll
            for (int k = 0; k < NP; ++k) tc::tmem_st_32x32b_x16(a0 + (uint32_t)k * ap + lanes + (uint32_t)(16 * cc), pc[k]);
        }
        tc::tmem_wait_st();
    }
    if (a.h_n) {
        for (int idx = threadIdx.x; idx < S * kCU; idx += kCT) {
            const int j = idx / kCU, uu = idx - j * kCU;
            if (j0 + j < a.B && s_len[j] == 0) {        // an empty sequence ends in its initial state
                const size_t o = ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + uu;
                a.h_n[o] = a.h0 ? a.h0[o] : 0.f;
                if (a.c_n) a.c_n[o] = a.c0 ? a.c0[o] : 0.f;
            }
        }
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    // tma_pre: the four gate tiles of step s2 (rows from off[t2], NBM of them; rows past the
    // packed rows read 0), one thread, completing on pre_bar.  The tiles of step s2 + kTileAhead
    // are brought into L2 at the same time, so that each load finds its rows there
    auto prefetch_pre = [&](int s2) {
        if (s2 >= Tg) return;
        const int t2 = dir == 0 ? s2 : Tg - 1 - s2;
#pragma unroll
        for (int g = 0; g < 4; ++g) tc::tma_prefetch_2d(&pre_map, dir * 4 * H + g * H + u0, s_off[t2]);
    };
    auto issue_pre = [&](int s2, bool fence) {
        const int t2 = dir == 0 ? s2 : Tg - 1 - s2;
        if (fence) fence_proxy_async_cta();
        tc::mbar_arrive_expect_tx(pre_bar, (uint32_t)(4 * NBM * kCU * 4));
#pragma unroll
        for (int g = 0; g < 4; ++g)
            tc::tma_load_2d(pre_tile + (size_t)g * NBM * kCU, &pre_map, pre_bar, dir * 4 * H + g * H + u0, s_off[t2]);
        prefetch_pre(s2 + kTileAhead);
    };
    int last_tile = -1;                   // tile issuer: the last step whose tile was issued
    if (tma_pre && threadIdx.x == kTileIssuer && Tg > 0) {
        for (int s2 = 1; s2 < kTileAhead; ++s2) prefetch_pre(s2);
        issue_pre(0, true);
        last_tile = 0;
    }
    cl.sync();     // every CTA of the cluster is resident before any remote write

    // cell item: row jq (+ RPP k), units uq .. uq + U: U units a thread, 32 / U threads a row
    constexpr int CPR = 32 / U, RPP = kCT / CPR, PASSES = 128 / RPP;
    const int jq = threadIdx.x / CPR, qc = threadIdx.x % CPR, uq = qc * U;
    using PkT = typename PkU<U>::T;
    const int nks = (H + 15) / 16;                                   // MMA k-steps
    float pk[3][U];                                                  // peepholes i, f, o of units uq .. + U
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
        for (int e = 0; e < U; ++e) pk[q][e] = peep_s[q * kCU + uq + e];
    const uint32_t bstep = (uint32_t)(NBM * (BULK ? 64 : 128)) >> 4;  // descriptor units between B blocks
    bool failed = false;                  // CTA-uniform: an MMA completion wait timed out
    bool pre_ok_prev = true;              // this thread's wait for the previous step's tile
    for (int s = 0; s < Tg; ++s) {
        const int t = dir == 0 ? s : Tg - 1 - s;
        const int n = s_bs[t];
        const int rowbase = s_off[t];
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < Tg ? s_bs[t + 1] : 0);
        const int NBs = (n + 15) & ~15;
        const int par = BULK ? (s & 1) : 0;
        bool arrived = true;          // this step's operand (and the previous step's tile) arrived
        if (BULK) {
            cstamp(a, false, dir, srank, s, 0, 0);
            // h_{t-1} of every peer has arrived in this step's operand
            if (s > 0 && !failed)
                arrived = tc::mbar_wait(&full_bar[par], (uint32_t)(((s - 1) >> 1) & 1), a.wait_limit_ns);
        } else {
            if (s > 0) {
                cluster_wait();    // h_{t-1} of every peer is in this CTA's operand
                // every thread of this CTA arrived after its cell: the tile is free
                if (tma_pre && threadIdx.x == kTileIssuer && !failed) { issue_pre(s, true); last_tile = s; }
                cstamp(a, false, dir, srank, s - 1, 4, 4);
            }
            cstamp(a, false, dir, srank, s, 0, 0);
        }
        // D[gate rows][rows] = R_slice x h_{t-1}^T: chain ch is issued by warp ch into its own
        // accumulator, so the chains overlap
        if (lane == 0 && warp < nch && !failed) {
            fence_proxy_async_cta();
            tc::tc_fence_after_sync();
            cstamp(a, false, dir, srank, s, 1, 1);
            const uint32_t idesc = tc::idesc_bf16_f32(kCM, NBs);
            const uint64_t bp = (uint64_t)(bsz >> 4);                  // descriptor units between B pieces
            if (BULK) {
                const uint64_t db0 = sdesc_sw64(tc::smem_u32(Bop(par, 0)));
                issue_chains32<NP>(nch, tmem + (uint32_t)(warp * NBM), a0, ap, db0, bp, bstep, nks, warp, idesc);
            } else {
                const uint64_t db0 = tc::sdesc_sw128(tc::smem_u32(Bop(0, 0)));
                issue_chains<NP>(nch, tmem + (uint32_t)(warp * NBM), a0, ap, db0, bp, bstep, nks, warp, idesc);
            }
            if (!(s == 0 && dir == 0 && grp == 0 && rank == a.debug_skip_cta)) tc::mma_commit(mma_bar);   // test hook
        }
        if (warp < nch) __syncwarp();     // the issuing lane's warp does not poll while it issues
        cstamp(a, false, dir, srank, s, 6, 6);
        // meanwhile (without tma_pre): the cell items' own operands (gate pre-activations),
        // rows jq and jq + RPP
        float pre[2][4][U];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int j = jq + it * RPP;
            if (!tma_pre && j < n) {
                const float* gr = a.ga + (size_t)(rowbase + j) * nd4H + dir * 4 * H + u0 + uq;
#pragma unroll
                for (int g = 0; g < 4; ++g) ld_u<U>(gr + g * H, pre[it][g]);
            }
        }
        if (!tma_pre && s + 1 < Tg) {   // next step's own rows into L2 (4 gate blocks of this CTA's units)
            const int t2 = dir == 0 ? s + 1 : Tg - 2 - s;
            for (int g = 0; g < 4; ++g)
                prefetch_rows(a.ga, nd4H, s_off[t2], s_bs[t2], dir * 4 * H + g * H + u0);
        }
        // A timeout (of the product, or of the operand's arrival) becomes a CTA-uniform decision
        // at the barrier after the read-out: from then on the CTA issues no product, waits for
        // no operand, re-arms nothing and sends nothing (so no barrier is armed twice and
        // unmatched bytes stay within two steps), and the teardown waits for the product in
        // flight before freeing tensor memory.  The read-out of the failing step itself may see
        // partial sums; the status word marks the results as invalid.
        const bool ok = failed ? true : tc::mbar_wait(mma_bar, (uint32_t)(s & 1), a.wait_limit_ns);
        arrived = arrived && pre_ok_prev;
        if ((!ok || !arrived) && !failed) {
            record_failure(a.status, LSTM_ERR_TIMEOUT, (ok ? 0x60000u : 0x40000u) | (unsigned)s);
            *s_fail = 1 + s;
        }
        cstamp(a, false, dir, srank, s, 7, 7);
        tc::tc_fence_after_sync();
        if (!BULK) cluster_arrive_relaxed();   // this CTA's product has read its operand: peers may overwrite it
        // accumulators -> shared: warp (quarter q = gate, half) reads lanes 32q.. in 16-column blocks
        if (!failed) {
            const int q = warp & 3, half = warp >> 2;
            for (int c0 = half * 16; c0 < NBs; c0 += 32) {
                float v[16];
                tmem_sum_chains(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, (uint32_t)NBM, nch, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) accs[(size_t)(c0 + e) * kCM + q * 32 + lane] = v[e];
            }
        }
        tc::tc_fence_before_sync();
        if (__syncthreads_or(!ok || !arrived)) failed = true;
        // BULK: re-arm this parity for step s + 2 before this CTA's h_t goes out (a peer
        // needs h_t before it can send h_{t+1})
        if (BULK && threadIdx.x == 0 && !failed && s + 2 < Tg)
            tc::mbar_arrive_expect_tx(&full_bar[par], step_bytes(s + 2));
        cstamp(a, false, dir, srank, s, 2, 2);
        // cell: row j, units u0 + uq .. + U; h_t kept (split) for the exchange.  Without the bulk
        // exchange the global outputs of rows jq and jq + RPP are written after the exchange's
        // barrier arrival, so that the arrival (a release) does not wait for them
        bool pre_ok = true;
        if (tma_pre && !failed) pre_ok = tc::mbar_wait(pre_bar, (uint32_t)(s & 1), a.wait_limit_ns);
        if (!pre_ok && !failed) {
            record_failure(a.status, LSTM_ERR_TIMEOUT, 0x70000u | (unsigned)s);
            *s_fail = 1 + s;
        }
        PkT xp[PASSES][NP];
        float og_[2][4][U], oc_[2][U], oh_[2][U];
        auto store_outputs = [&](int j, const float (&gg)[4][U], const float (&cv)[U], const float (&hv)[U],
                                 PkT hi) {
            const int row = rowbase + j;
            const int len = s_len[j];
            float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + uq;
#pragma unroll
            for (int g = 0; g < 4; ++g) st_u<U>(gr + g * H, gg[g]);
            const size_t yo = (size_t)row * ndH + dir * H + u0 + uq;
            st_u<U>(a.cbuf + yo, cv);
            st_u<U>(a.y + yo, hv);
            if (a.y_lo) *reinterpret_cast<PkT*>(a.y_lo + yo) = hi;
            if (a.h_n && ((dir == 0 && t == len - 1) || (dir == 1 && t == 0 && len > 0))) {
                const size_t o = ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + uq;
#pragma unroll
                for (int e = 0; e < U; ++e) {
                    a.h_n[o + e] = hv[e];
                    if (a.c_n) a.c_n[o + e] = cv[e];
                }
            }
        };
#pragma unroll
        for (int it = 0; it < PASSES; ++it) {
            const int j = jq + it * RPP;
            if (j >= n) continue;
            const int len = s_len[j];
            float pv[4][U];
            if (tma_pre) {
#pragma unroll
                for (int g = 0; g < 4; ++g) ld_u<U>(pre_tile + ((size_t)g * NBM + j) * kCU + uq, pv[g]);
            } else if (it < 2) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int e = 0; e < U; ++e) pv[g][e] = it == 0 ? pre[0][g][e] : pre[1][g][e];
            } else {
                const float* gr = a.ga + (size_t)(rowbase + j) * nd4H + dir * 4 * H + u0 + uq;
#pragma unroll
                for (int g = 0; g < 4; ++g) ld_u<U>(gr + g * H, pv[g]);
            }
            float hv[U], cv[U], gg[4][U];
            // the row's products of the 4 gates and its previous cell states, U units at a time
            float acv[4][U], cpv[U];
#pragma unroll
            for (int g = 0; g < 4; ++g) ld_u<U>(accs + (size_t)j * kCM + g * kCU + uq, acv[g]);
            if (j < n_prev) {
                ld_u<U>(cst + j * kCU + uq, cpv);
            } else if (a.c0) {
                ldg_u<U>(a.c0 + ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + uq, cpv);
            } else {
#pragma unroll
                for (int e = 0; e < U; ++e) cpv[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < U; ++e) {
                const float cp = cpv[e];
                const float ig = sigm_c(pv[0][e] + acv[0][e] + pk[0][e] * cp);
                const float fg = sigm_c(pv[1][e] + acv[1][e] + pk[1][e] * cp);
                const float zg = tanh_c(pv[2][e] + acv[2][e]);
                float c = fg * cp + ig * zg;
                const float og = sigm_c(pv[3][e] + acv[3][e] + pk[2][e] * c);
                float h = og * tanh_c(c);
                if (a.padded && t >= len) { c = 0.f; h = 0.f; }
                gg[0][e] = ig; gg[1][e] = fg; gg[2][e] = zg; gg[3][e] = og; cv[e] = c; hv[e] = h;
            }
            st_u<U>(cst + j * kCU + uq, cv);
            split_u<U, NP>(hv, xp[it]);
            if (!BULK && it < 2) {
#pragma unroll
                for (int e = 0; e < U; ++e) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) og_[it][g][e] = gg[g][e];
                    oc_[it][e] = cv[e];
                    oh_[it][e] = hv[e];
                }
            } else {
                store_outputs(j, gg, cv, hv, xp[it][0]);
            }
        }
        cstamp(a, false, dir, srank, s, 5, 5);
        if (BULK) {
            // h_t (rows [0, NBs)) staged in this CTA's 32-unit block, then one bulk copy per peer
            // and half into that peer's operand of step s + 1
            if (s + 1 < Tg) {
#pragma unroll
                for (int it = 0; it < PASSES; ++it) {
                    const int j = jq + it * RPP;
                    if (j >= n) continue;
                    const uint32_t o = sw64_off_u<U>(j, qc);
                    // this CTA's own block of the next step's operand is written in place
                    const size_t ob = (size_t)rank * NBM * 64 + o;
#pragma unroll
                    for (int k = 0; k < NP; ++k) {
                        *reinterpret_cast<PkT*>(Stg(par, k) + o) = xp[it][k];
                        *reinterpret_cast<PkT*>(Bop(par ^ 1, k) + ob) = xp[it][k];
                    }
                }
            }
            fence_proxy_async_cta();
            __syncthreads();
            // lane 0 of warp w sends to peers w, w + 8 (copies issued by one warp's lanes serialise)
            const bool sender = lane == 0 && warp < G;
            if (s + 1 < Tg && sender && !failed) {
                const uint32_t nxt = (uint32_t)(par ^ 1);
                const uint32_t bytes = (uint32_t)step_rows(s + 1) * 64u;
                for (int p2 = warp; p2 < G; p2 += kCT / 32) {
                    if (p2 == (int)rank || bytes == 0) continue;
                    const uint32_t bar = mapa_u32(tc::smem_u32(&full_bar[nxt]), (uint32_t)p2);
#pragma unroll
                    for (int k = 0; k < NP; ++k)
                        bulk_to_peer(mapa_u32(tc::smem_u32(Bop(nxt, k) + (size_t)rank * NBM * 64), (uint32_t)p2),
                                     Stg(par, k), bytes, bar);
                }
                bulk_commit();
            }
            cstamp(a, false, dir, srank, s, 4, 4);
            if (tma_pre && threadIdx.x == kTileIssuer && s + 1 < Tg && !failed) {   // the tile has been read
                issue_pre(s + 1, false);
                last_tile = s + 1;
            }
            if (s + 1 < Tg && sender && !failed) bulk_wait_read_all_but_one();   // step s - 1's staging
        } else {
            cluster_wait();        // every peer's product of this step is done with its operand
            // h_t into every peer's operand of the next step (row j, columns u0 + uq ..)
            if (s + 1 < Tg) {
#pragma unroll
                for (int it = 0; it < PASSES; ++it) {
                    const int j = jq + it * RPP;
                    if (j >= n) continue;
                    const uint32_t o = sw_off4(j, u0 + uq, NBM);
                    for (int p2 = 0; p2 < G; ++p2)
#pragma unroll
                        for (int k = 0; k < NP; ++k)
                            *reinterpret_cast<PkT*>(cl.map_shared_rank(Bop(0, k) + o, p2)) = xp[it][k];
                }
            }
            fence_proxy_async_cluster();
            cluster_arrive();      // release: this CTA's h_t is in every peer's operand
        }
        if (!BULK) {
#pragma unroll
            for (int it = 0; it < 2; ++it)
                if (jq + it * RPP < n) store_outputs(jq + it * RPP, og_[it], oc_[it], oh_[it], xp[it][0]);
        }
        pre_ok_prev = pre_ok;
        cstamp(a, false, dir, srank, s, 3, 3);
    }
    // after a timeout the last tile issued may not have been waited for: no load may still be
    // writing this CTA's shared memory when it exits (bounded wait)
    if (tma_pre && threadIdx.x == kTileIssuer && last_tile >= 0)
        tc::mbar_wait(pre_bar, (uint32_t)(last_tile & 1), kTeardownWaitNs);
    if (BULK) {
        if (lane == 0 && warp < G) bulk_wait_all();   // no copy of this CTA is still in flight
        cl.sync();                              // nor one into it: every CTA has passed its last wait
    } else if (Tg > 0) {
        cluster_wait();            // the last step's arrival
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

// ------------------------------------------------------------------------- configuration
template <int U>
static const void* fwd_kernel_u(bool bf16, bool bulk)
{
    if (bulk) return bf16 ? (const void*)lstm_rec_fwd_cluster_kernel<1, true, U>
                          : (const void*)lstm_rec_fwd_cluster_kernel<3, true, U>;
    return bf16 ? (const void*)lstm_rec_fwd_cluster_kernel<1, false, U> : (const void*)lstm_rec_fwd_cluster_kernel<3, false, U>;
}
static const void* fwd_kernel(bool bf16, bool bulk, int group_rows)
{
    return cell_units(group_rows, false) == 2 ? fwd_kernel_u<2>(bf16, bulk) : fwd_kernel_u<4>(bf16, bulk);
}

bool rec_cluster_fwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* lay)
{
    if (p.gemm_engine != 0 || p.forced_ctas != 0) return false;
    if (H % kCU != 0) return false;
    const int G = H / kCU;
    if (G > 16 || G * ndir > p.num_sms) return false;
    int S = 0, ng = 1;
    if (!choose_groups(p, G, ndir, &S, &ng)) return false;
    const int NBM = std::max(16, (std::min(S, max_active_rows(p)) + 15) & ~15);
    const int np = bf16 ? 1 : 3;                   // bf16 pieces of each operand
    const int KB = (H + 63) / 64;
    const int nks = (H + 15) / 16;
    const int acols = (H / 2) * np;                // R slice in TMEM, two bf16 per column and piece
    int nch = 4;
    while (nch > 1 && (nch > nks || nch * NBM + acols > 512)) nch >>= 1;
    if (nch * NBM + acols > 512) return false;
    const uint32_t cols = pow2_cols(nch * NBM + acols);
    // preference: TMA pre-activation tiles, then the bulk exchange (double-buffered operand +
    // staging); the single-buffered exchange without tiles needs the least shared memory
    const int order[4][2] = {{1, 1}, {0, 1}, {1, 0}, {0, 0}};
    for (int oi = 0; oi < 4; ++oi) {
        const int bulk = order[oi][0], pre = order[oi][1];
        if (p.forced_variant >= 0 && p.forced_variant != (bulk | pre << 1)) continue;
        const size_t bbytes = bulk ? 2 * (size_t)np * G * NBM * 64 : (size_t)np * KB * NBM * 128;
        size_t off = 0;
        const size_t o_b = off; off = al(off + bbytes, 1024);
        const size_t o_stage = off; if (bulk) off = al(off + 2 * (size_t)np * NBM * 64, 1024);
        const size_t o_pre = off; if (pre) off = al(off + 4 * (size_t)NBM * kCU * 4, 1024);
        const size_t o_acc = off; off = al(off + (size_t)NBM * kCM * 4, 16);
        const size_t o_cst = off; off = al(off + (size_t)S * kCU * 4, 16);
        const size_t o_bar = off; off = al(off + 64, 16);
        const size_t o_peep = off; off = al(off + 3 * kCU * 4, 16);
        const size_t o_tab = off; off = al(off + (size_t)(2 * p.T + 1 + S) * 4, 16);
        size_t smem = off + 1024 + 64;            // 1024 for the base alignment, 64 static
        smem = tmem_safe_smem(p, smem, cols);
        if (smem == 0) return false;
        if (!cluster_schedulable(p, fwd_kernel(bf16, bulk != 0, S), G, smem)) continue;
        RecConfig c;
        c.G = G; c.Umax = (int)cols; c.JC = NBM; c.smem = smem; c.cluster = 1;
        c.chains = nch; c.acol = (int)cols - acols; c.bulk = bulk; c.tma_pre = pre;
        c.grp_rows = S; c.ngroups = ng;
        *out = c;
        lay->off_contrib = (int)o_b; lay->off_h = (int)o_stage; lay->off_red = (int)o_pre; lay->off_acc = (int)o_acc;
        lay->off_state = (int)o_cst; lay->off_sums = (int)o_bar; lay->off_peep = (int)o_peep;
        lay->off_tab = (int)o_tab;
        return true;
    }
    return false;
}

lstm_status rec_cluster_fwd_launch(const Plan& p, const RecConfig& c, RecArgs a, cudaStream_t s)
{
    a.G = c.G; a.Umax = c.Umax; a.JC = c.JC; a.tm_chains = c.chains; a.tm_acol = c.acol;
    a.grp_rows = c.grp_rows; a.ngroups = c.ngroups;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    const void* fn = fwd_kernel(a.bf16 != 0, c.bulk != 0, c.grp_rows);
    // the pre-activation tiles' map: ga as [rows][ndir*4H] fp32, boxes of 32 units x NBM rows
    CUtensorMap pre_map;
    memset(&pre_map, 0, sizeof(pre_map));
    const int nd4H = a.ndir * 4 * a.H;
    a.tma_pre = c.tma_pre && make_map_f32(&pre_map, a.ga, p.rows, nd4H, nd4H, kCU, c.JC) ? 1 : 0;
    void* args[] = {&a, &pre_map};
    trace_begin(p, K_REC_FWD, s);
    const lstm_status st = cluster_launch(c, fn, args, a.ndir, s);
    trace_end(p, K_REC_FWD, s, st == LSTM_OK ? 1 : 0);
    return st;
}

}  // namespace lstm
