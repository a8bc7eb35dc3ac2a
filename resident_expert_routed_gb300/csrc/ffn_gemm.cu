// Grouped expert GEMMs over the MXFP4 slot arena on the 5th-generation tensor
// cores (tcgen05, kind::mxf4 block-scaled MMA, accumulators in TMEM).
//
// TideLM README: the experts are "native MXFP4" (profile table) and live in
// one arena of slots shared by all layers (item 1); the picks of a step are
// routed only to resident slots (item 2). One launch per GEMM covers every
// used slot: the work list from ffn_plan names (slot, first row, rows) tiles.
//
//   gate/up (MODE 1): for 128 ffn features f0..f0+127 of one slot, two MMAs
//       per K step, D_g = Wg[f0..] x A and D_u = Wu[f0..] x A (M 128 each, N =
//       the tile's activation rows, K = d) into two TMEM accumulators; the
//       epilogue thread of TMEM lane f holds g and u of feature f0 + f, forms
//       h = silu(g) * u and re-quantises it to MXFP4 in blocks of 32 features
//       (one warp = one block; OCP MX v1.0 rule) into the down GEMM's operand.
//   down (MODE 2): for 128 output rows d0..d0+127, D = Wd rows x hq rows,
//       K = ffn; epilogue: fp32 rows Y[pick] (combined later in pick order).
//
// The weight tiles are the MMA's A operand (M = 128) and the few routed rows
// the B operand (N = 16..128), so a decode-sized tile still streams whole
// weight tiles at full width. Roles:
//   warp 4     lane 0, per stage: 64 KB of weight codes as contiguous bulk
//              copies (the arena keeps codes in tile-major 16 KB blocks, already
//              in the 128-byte swizzle) and TMA boxes of activation rows (their
//              height the tile's row count rounded up);
//   warps 6-9  scale factors: each warp (one TMEM lane quadrant) loads the
//              stage's scale atoms (weights: from the arena, which keeps them in
//              the tensor cores' atom order; activations: from the workspace,
//              written in that order by ffn_pack / the gate/up epilogue) and
//              writes them into TMEM with tcgen05.st (see scale_writer);
//   warp 5     TMEM allocator; lane 0 issues tcgen05.mma and commits to the
//              stage / accumulator barriers;
//   warps 0-3  epilogue: tcgen05.ld of their 32-lane quadrant of the
//              (double-buffered) accumulators, then the per-mode epilogue.
// The grid is persistent (one CTA per SM) over the flattened (tile, 128-row
// weight block) items. Every wait is bounded (the host's moe_set_wait_limit,
// 2 s by default); on expiry the CTA raises its abort flag, every role leaves
// its loop, the producer waits for the bytes of the copies it has issued and
// the MMA thread for its MMAs, TMEM is freed and the device error word gets
// MOE_DEV_TIMEOUT.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace {

struct GemmMaps {
    CUtensorMap b[4];     // activation codes: (row bytes, positions), box 128 B x {16, 32, 64, 128} rows
};

struct GemmArgs {
    const uint8_t* arena;
    int64_t slot_bytes;
    int64_t off_codes;           // this GEMM's weight codes within a slot (tile-major 16 KB blocks)
    int64_t off_scales;          // this GEMM's weight scales within a slot (tile-atom order)
    int K;                       // reduction length: d (gate/up) or ffn (down)
    int m_tiles;
    int F;                       // ffn
    int d;                       // hidden size
    const int4* work;
    const int32_t* n_work;
    const int32_t* pair_of_pos;
    const uint8_t* b_scales;     // activation scale atoms (xsp or hsp)
    uint8_t* hq;                 // gate/up output: down activation codes [pad_max, F/2]
    uint8_t* hsp;                // gate/up output: down activation scale atoms
    float* Y;                    // down output [T*k, d] (per-pick rows)
    uint32_t* err;
    uint64_t wait_ns;            // bound on each pipeline wait
    int evict_first;             // weights read once (decode tiles): stream them with an L2 evict-first policy
};

// Scale factors reach TMEM through registers, not tcgen05.cp: the copy that
// replicates a 32-row atom into the four TMEM lane quadrants occupies the
// tensor pipe for about half an MMA, and a stage needs one per 128 K of every
// operand. Warps 6-9 (one per lane quadrant) instead load each stage's atoms
// from global memory PF stages ahead and write them with tcgen05.st, which
// runs beside the MMAs; they signal the MMA thread through sfull[stage]. Lane
// i of every quadrant holds row i (16 bytes) of each 512-byte atom, the layout
// the 32x128b.warpx4 copy produces. load(g, v) fills the NV atoms of stage g
// (zeros past the end of K).
template <int NV, int PF, int NS, typename Load>
__device__ __forceinline__ void scale_writer(int n_stages, const Load& load, uint64_t* empty, uint64_t* sfull,
                                             uint32_t sf_base, int sf_cols, volatile int* abort_flag,
                                             uint64_t wait_ns) {
    static_assert(NV % 2 == 0, "atoms are written in pairs");
    const int lane = threadIdx.x & 31;
    uint4 v[PF][NV];
#pragma unroll
    for (int p = 0; p < PF; ++p) load(p, v[p]);
    bool ok_run = true;
    for (int g0 = 0; g0 < n_stages && ok_run; g0 += PF) {
#pragma unroll
        for (int p = 0; p < PF; ++p) {
            const int g = g0 + p;
            if (g >= n_stages) break;
            const int s = g % NS;
            const uint32_t r = (uint32_t)(g / NS);
            if (!warp_wait(&empty[s], (r & 1) ^ 1, abort_flag, wait_ns)) { ok_run = false; break; }
            tc_fence_after();
            const uint32_t sfc = sf_base + s * sf_cols;
#pragma unroll
            for (int q = 0; q < NV; q += 2) tc_st_x8(sfc + 4 * q, v[p][q], v[p][q + 1]);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfull[s]);
            load(g + PF, v[p]);
        }
    }
}

// The same hand-off with the scale atoms staged in shared memory: the
// producer copies each stage's atoms with bulk copies that complete on a
// barrier of the stage (`full`, or in the token-major kernel a barrier of
// their own, issued before the operands, so that the writers fill TMEM while
// the 48 KB of operands are still arriving), so their global latency is hidden
// by the copy pipeline like the operands' (loading them from global memory in
// the writer warps, even four stages ahead, left the MMA thread waiting ~260
// cycles per stage on the 8192-token gate/up GEMM). Per stage: wait for the
// atoms, read this lane's 16-byte row of each (atom v[q] at smem atom slot
// `slot_of_atom(q)`; atoms past the end of K are zeros), write them into
// TMEM, tell the MMA thread. The TMEM columns of a stage are free by then: the
// producer refilled the stage only after the MMAs that read them completed.
template <int NV, int NS, typename Valid, typename Slot>
__device__ __forceinline__ void scale_writer_smem(int n_stages, const Valid& valid, const Slot& slot_of_atom,
                                                  uint64_t* full, uint64_t* sfull, const uint8_t* sf_smem,
                                                  int sf_stage_bytes, uint32_t sf_base, int sf_cols,
                                                  volatile int* abort_flag, uint64_t wait_ns) {
    static_assert(NV % 2 == 0, "atoms are written in pairs");
    const int lane = threadIdx.x & 31;
    for (int g = 0; g < n_stages; ++g) {
        const int s = g % NS;
        const uint32_t r = (uint32_t)(g / NS);
        if (!warp_wait(&full[s], r & 1, abort_flag, wait_ns)) break;
        const uint8_t* src = sf_smem + s * sf_stage_bytes + lane * 16;
        const int nvalid = valid(g);
        uint4 v[NV];
#pragma unroll
        for (int q = 0; q < NV; ++q)
            v[q] = slot_of_atom(q, nvalid) >= 0 ? *reinterpret_cast<const uint4*>(src + slot_of_atom(q, nvalid) * 512)
                                                : make_uint4(0u, 0u, 0u, 0u);
        tc_fence_after();
        const uint32_t sfc = sf_base + s * sf_cols;
#pragma unroll
        for (int q = 0; q < NV; q += 2) tc_st_x8(sfc + 4 * q, v[q], v[q + 1]);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[s]);
    }
}

// Per pipeline stage: KCH chunks of 256 elements along K. The gate/up GEMM
// loads, per chunk, one 16 KB code block of the gate tile and one of the up
// tile (rows f0..f0+127 and ffn+f0..ffn+f0+127) and accumulates them into two
// TMEM accumulators, so that each epilogue thread holds g and u of the same
// feature; the down GEMM loads one tile. Decode stages carry 64 KB of weights
// (two chunks of gate and up, or four of one down tile); with twice the atoms
// per stage the scale writers then look two stages ahead instead of four.
template <int MODE, int BN, int NS, int KCH, int NBUF, bool STAGED = false>
struct Cfg {
    static constexpr int THREADS = 320;           // warps 0-3 epilogue, 4 TMA, 5 MMA, 6-9 scales
    static constexpr int NMAT = MODE == 1 ? 2 : 1;
    static constexpr int BLK = 128 * 128;         // one 16 KB code block: 128 rows x 256 e2m1
    static constexpr int A_BYTES = NMAT * KCH * BLK;
    static constexpr int B_CHUNK = BN * 128;
    static constexpr int B_BYTES = KCH * B_CHUNK;
    static constexpr int NV = (NMAT + 1) * 2 * KCH;        // scale atoms per stage (weights, then activations)
    static constexpr int PF = NMAT * KCH >= 4 ? 2 : 4;     // stages of scales loaded ahead (registers: PF NV uint4)
    static_assert(PF >= 1, "scale look-ahead");
    static constexpr int SF_COLS = 4 * NV;                 // TMEM columns of one stage's scales
    static constexpr int ACC_COLS = NMAT * BN;    // one accumulator buffer (gate, then up)
    // STAGED: each stage's scale atoms are copied into shared memory by the producer (weights first,
    // then the activations', as in the register order) instead of loaded by the writer warps
    static constexpr int SF_STAGE = STAGED ? NV * 512 : 0;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + NS * A_BYTES;
    static constexpr int OFF_SF = OFF_B + NS * B_BYTES;
    static constexpr int OFF_BAR = OFF_SF + NS * SF_STAGE;
    // full, empty, sfull (and, staged, satoms: the scale atoms alone) per stage; accf, acce; drain
    static constexpr int N_BARS = (STAGED ? 4 : 3) * NS + 2 * NBUF + 1;
    static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;   // + slack to align the base to 1024
    static constexpr int TMEM_USED = NBUF * ACC_COLS + SF_COLS * NS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256 : 512;
    static_assert(BN == 16 || BN == 32 || BN == 64 || BN == 128, "BN");
    static_assert(KCH == 1 || KCH == 2 || KCH == 4, "KCH");
    static_assert(NBUF == 1 || NBUF == 2, "NBUF");
    static_assert(TMEM_USED <= 512, "TMEM");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int MODE, int BN, int NS, int KCH, int NBUF, bool STAGED>
__global__ void __launch_bounds__(320, 1) ffn_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    using C = Cfg<MODE, BN, NS, KCH, NBUF, STAGED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + NS;
    uint64_t* sfull = empty + NS;
    uint64_t* satoms = sfull + NS;                   // staged: the stage's scale atoms (the writers' wait)
    uint64_t* accf = satoms + (STAGED ? NS : 0);
    uint64_t* acce = accf + NBUF;
    uint64_t* drain = acce + NBUF;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1); mbar_init(&empty[s], 1); mbar_init(&sfull[s], 4);
            if (STAGED) mbar_init(&satoms[s], 1);
        }
        for (int b = 0; b < NBUF; ++b) { mbar_init(&accf[b], 1); mbar_init(&acce[b], 4); }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        for (int i = 0; i < 4; ++i) prefetch_tmap(&maps.b[i]);
    }
    if (warp == 5) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    uint32_t issued = 0;                             // stage fills issued by the producer thread
    pdl_wait();                                      // the work list is the plan kernel's output
    const int n_items = *a.n_work * a.m_tiles;
    const int nc = (a.K + 255) / 256;                 // 256-element chunks along K
    const int nst = (nc + KCH - 1) / KCH;             // pipeline stages per item
    const int atoms = a.K / 128;                      // scale atoms per 128-row tile

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer (one thread)
        if (lane == 0) {
            uint32_t& it = issued;
            bool ok_run = true;
            const uint64_t policy = l2_evict_first_policy();
            int4 w_next = blockIdx.x < n_items ? a.work[blockIdx.x / a.m_tiles] : make_int4(0, 0, 0, 0);
            for (int item = blockIdx.x; item < n_items && ok_run; item += gridDim.x) {
                const int4 w = w_next;
                const int nxt = item + gridDim.x;          // fetch the next entry while this item streams
                if (nxt < n_items) w_next = a.work[nxt / a.m_tiles];
                const int mt = item % a.m_tiles;
                const int slot = w.x, pos0 = w.y, nv = w.z;
                const int hb = nv <= 16 ? 0 : nv <= 32 ? 1 : nv <= 64 ? 2 : 3;   // activation box height
                const uint32_t b_bytes = (16u << hb) * 128u;
                const uint8_t* rec = a.arena + (size_t)slot * a.slot_bytes;
                // weight tiles: gate mt and up F/128 + mt, or down mt
                const int tile0 = mt, tile1 = a.F / 128 + mt;
                const uint8_t* codes0 = rec + a.off_codes + (size_t)tile0 * nc * C::BLK;
                const uint8_t* codes1 = rec + a.off_codes + (size_t)tile1 * nc * C::BLK;
                for (int st = 0; st < nst; ++st, ++it) {
                    const int s = (int)(it % NS);
                    const uint32_t r = it / NS;
                    if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, a.wait_ns)) { ok_run = false; break; }
                    uint8_t* As = smem + C::OFF_A + s * C::A_BYTES;
                    uint8_t* Bs = smem + C::OFF_B + s * C::B_BYTES;
                    const int c0 = st * KCH;
                    const int chunks = nc - c0 < KCH ? nc - c0 : KCH;
                    uint32_t sf_bytes = 0;
                    if constexpr (STAGED) {
                        // the scale atoms first, on their own barrier: the writers move them into TMEM while
                        // the stage's 64 KB of weights are still arriving
                        const int at0 = 2 * KCH * st;
                        sf_bytes = (uint32_t)(atoms - at0 < 2 * KCH ? atoms - at0 : 2 * KCH) * 512u;
                        uint8_t* Ss = smem + C::OFF_SF + s * C::SF_STAGE;
                        const size_t at0b = (size_t)at0 * 512;
                        const uint8_t* sc = rec + a.off_scales;
                        mbar_arrive_expect_tx(&satoms[s], (C::NMAT + 1) * sf_bytes);
                        bulk_load(Ss, sc + (size_t)tile0 * atoms * 512 + at0b, sf_bytes, &satoms[s]);
                        if (C::NMAT == 2)
                            bulk_load(Ss + 2 * KCH * 512, sc + (size_t)tile1 * atoms * 512 + at0b, sf_bytes,
                                      &satoms[s]);
                        bulk_load(Ss + C::NMAT * 2 * KCH * 512, a.b_scales + (size_t)(pos0 / BN) * atoms * 512 + at0b,
                                  sf_bytes, &satoms[s]);
                    }
                    mbar_arrive_expect_tx(&full[s], (uint32_t)chunks * (C::NMAT * C::BLK + b_bytes));
                    if (a.evict_first) {
                        bulk_load_hint(As, codes0 + (size_t)c0 * C::BLK, (uint32_t)chunks * C::BLK, &full[s], policy);
                        if (C::NMAT == 2)
                            bulk_load_hint(As + KCH * C::BLK, codes1 + (size_t)c0 * C::BLK, (uint32_t)chunks * C::BLK,
                                           &full[s], policy);
                    } else {
                        bulk_load(As, codes0 + (size_t)c0 * C::BLK, (uint32_t)chunks * C::BLK, &full[s]);
                        if (C::NMAT == 2)
                            bulk_load(As + KCH * C::BLK, codes1 + (size_t)c0 * C::BLK, (uint32_t)chunks * C::BLK,
                                      &full[s]);
                    }
                    for (int q = 0; q < chunks; ++q)
                        tma_load_2d(Bs + q * C::B_CHUNK, &maps.b[hb], &full[s], (c0 + q) * 128, pos0);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // One thread feeds the tensor pipe, which queues few MMAs, so the loop
            // keeps its per-stage work small: descriptors offset from per-kernel
            // bases (a K step of 32 bytes adds 2 to the address field, which cannot
            // carry below 256 KB of shared memory), stage and phase counters, the
            // row count of the next item loaded one item ahead.
            int s = 0;
            uint32_t ph = 0, j = 0;
            bool ok_run = true;
            const uint64_t a_base = smem_desc_sw128(smem_u32(smem + C::OFF_A));
            const uint64_t b_base = smem_desc_sw128(smem_u32(smem + C::OFF_B));
            const uint32_t sf_base = tmem + NBUF * C::ACC_COLS;
            int nv_next = blockIdx.x < n_items ? a.work[blockIdx.x / a.m_tiles].z : 0;
            for (int item = blockIdx.x; item < n_items && ok_run; item += gridDim.x, ++j) {
                const int nv = nv_next;
                if (item + (int)gridDim.x < n_items) nv_next = a.work[(item + gridDim.x) / a.m_tiles].z;
                const int N = (nv + 15) & ~15;
                const uint32_t id0 = idesc_mxf4(N, 0, 0), id1 = idesc_mxf4(N, 2, 2);
                const int b = (int)(j % NBUF);
                const uint32_t u = j / NBUF;
                if (!mbar_wait(&acce[b], (u & 1) ^ 1, abort_flag, a.wait_ns)) break;
                tc_fence_after();
                const uint32_t dt = tmem + b * C::ACC_COLS;
                for (int st = 0; st < nst; ++st) {
                    if (!mbar_wait(&full[s], ph, abort_flag, a.wait_ns) || !mbar_wait(&sfull[s], ph, abort_flag, a.wait_ns)) {
                        ok_run = false;
                        break;
                    }
                    tc_fence_after();
                    const int rem = (a.K - st * 256 * KCH) / 64;
                    const int ksteps = rem < 4 * KCH ? rem : 4 * KCH;      // MMAs of K = 64
                    // scale columns: weight matrices m < NMAT, then activations, 8 KCH columns each
                    const uint32_t sfc = sf_base + s * C::SF_COLS;
                    const uint32_t sfb = sfc + 8 * KCH * C::NMAT;
                    const uint64_t ad = a_base + (uint32_t)(s * C::A_BYTES >> 4);
                    const uint64_t bd = b_base + (uint32_t)(s * C::B_BYTES >> 4);
                    if (ksteps == 4 * KCH) {
#pragma unroll
                        for (int kk = 0; kk < 4 * KCH; ++kk) {
                            const int q = kk >> 2, kq = kk & 3;
#pragma unroll
                            for (int m = 0; m < C::NMAT; ++m)
                                tc_mma_mxf4(dt + m * BN, ad + (((m * KCH + q) * C::BLK + kq * 32) >> 4),
                                            bd + ((q * C::B_CHUNK + kq * 32) >> 4), (kk & 1) ? id1 : id0,
                                            sfc + 8 * KCH * m + (kk >> 1) * 4, sfb + (kk >> 1) * 4,
                                            (st | kk) != 0 ? 1u : 0u);
                        }
                    } else {
                        for (int kk = 0; kk < ksteps; ++kk) {
                            const int q = kk >> 2, kq = kk & 3;
                            for (int m = 0; m < C::NMAT; ++m)
                                tc_mma_mxf4(dt + m * BN, ad + (((m * KCH + q) * C::BLK + kq * 32) >> 4),
                                            bd + ((q * C::B_CHUNK + kq * 32) >> 4), (kk & 1) ? id1 : id0,
                                            sfc + 8 * KCH * m + (kk >> 1) * 4, sfb + (kk >> 1) * 4,
                                            (st | kk) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(&empty[s]);
                    if (++s == NS) { s = 0; ph ^= 1; }
                }
                if (ok_run) tc_commit(&accf[b]);
            }
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------------ scale factors -> TMEM
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        auto load = [&](int g, uint4 (&v)[C::NV]) {
#pragma unroll
            for (int q = 0; q < C::NV; ++q) v[q] = make_uint4(0u, 0u, 0u, 0u);
            if (g >= my_items * nst) return;
            const int li = g / nst, st = g - li * nst;
            const int item = blockIdx.x + li * gridDim.x;
            const int wi = item / a.m_tiles;
            const int4 w = a.work[wi];
            const int mt = item - wi * a.m_tiles;
            const uint8_t* sc = a.arena + (size_t)w.x * a.slot_bytes + a.off_scales;
            const uint8_t* src[C::NMAT + 1];
            src[0] = sc + (size_t)mt * atoms * 512;
            if (C::NMAT == 2) src[1] = sc + (size_t)(a.F / 128 + mt) * atoms * 512;
            src[C::NMAT] = a.b_scales + (size_t)(w.y / BN) * atoms * 512;
            const int at0 = 2 * KCH * st;
            const int ats = atoms - at0 < 2 * KCH ? atoms - at0 : 2 * KCH;
#pragma unroll
            for (int m = 0; m <= C::NMAT; ++m)
#pragma unroll
                for (int q = 0; q < 2 * KCH; ++q)
                    if (q < ats)
                        v[m * 2 * KCH + q] =
                            *reinterpret_cast<const uint4*>(src[m] + (size_t)(at0 + q) * 512 + lane * 16);
        };
        const uint32_t sf_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + NBUF * C::ACC_COLS;
        if constexpr (STAGED) {
            // staged in register order: atom q of matrix m (weights first, then activations) at slot q
            auto valid = [&](int g) {
                const int at0 = 2 * KCH * (g % nst);
                return atoms - at0 < 2 * KCH ? atoms - at0 : 2 * KCH;
            };
            auto slot_of_atom = [](int q, int nvalid) { return (q % (2 * KCH)) < nvalid ? q : -1; };
            scale_writer_smem<C::NV, NS>(my_items * nst, valid, slot_of_atom, satoms, sfull, smem + C::OFF_SF,
                                         C::SF_STAGE, sf_base, C::SF_COLS, abort_flag, a.wait_ns);
        } else {
            scale_writer<C::NV, C::PF, NS>(my_items * nst, load, empty, sfull, sf_base, C::SF_COLS, abort_flag,
                                           a.wait_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0..3)
        // chk = fma(chk, 0, v) over every valid output: it stays finite while every value is finite and
        // turns NaN for good after a non-finite one (NaN * 0 and inf * 0 are NaN)
        float chk = 0.0f;
        uint32_t j = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
            const int4 w = a.work[item / a.m_tiles];
            const int mt = item % a.m_tiles;
            const int pos0 = w.y, nv = w.z;
            const int b = (int)(j % NBUF);
            const uint32_t u = j / NBUF;
            // down: the picks of the tile's columns, fetched before the accumulator is ready
            // (lane l holds column 32 q + l in pp[q])
            int pp[BN / 32 > 0 ? BN / 32 : 1];
            if (MODE == 2) {
#pragma unroll
                for (int q = 0; q * 32 < BN; ++q) {
                    const int col = q * 32 + lane;
                    pp[q] = col < nv ? a.pair_of_pos[pos0 + col] : 0;
                }
            }
            if (!warp_wait(&accf[b], u & 1, abort_flag, a.wait_ns)) break;
            tc_fence_after();
            const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16) + b * C::ACC_COLS;
            if (MODE == 1) {
                // lane of warp q holds gate and up of feature f0 + 32 q + lane: one 32-block per warp
                const int fb = mt * 128 + warp * 32;
                for (int c0 = 0; c0 < nv; c0 += 16) {
                    uint32_t vg[16], vu[16];
                    tc_ld_x16(trow + c0, vg);
                    tc_ld_x16(trow + BN + c0, vu);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (c0 + i >= nv) break;                 // warp-uniform
                        const float h = silu_mul(__uint_as_float(vg[i]), __uint_as_float(vu[i]));
                        chk = fmaf(chk, 0.0f, h);
                        float amax = fabsf(h);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1)
                            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
                        const int X = mx_shared_exp(amax);
                        const float hs = h * exp2_int(-X);
                        const float hs_hi = __shfl_down_sync(0xFFFFFFFFu, hs, 1);
                        const uint32_t byte = e2m1x2(hs, hs_hi);      // valid on even lanes
                        const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, byte, 2);
                        const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, byte, 4);
                        const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, byte, 6);
                        const int pos = pos0 + c0 + i;
                        if ((lane & 7) == 0)
                            *reinterpret_cast<uint32_t*>(a.hq + (size_t)pos * (a.F / 2) + fb / 2 + (lane >> 3) * 4) =
                                byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
                        if (lane == 0) a.hsp[operand_scale_offset(pos, fb / 32, BN, a.F)] = (uint8_t)(X + 127);
                    }
                }
            } else {
                // lane = output dim dr; each column is one pick: a warp stores 128 contiguous bytes of Y
                float* ycol = a.Y + mt * 128 + warp * 32 + lane;
#pragma unroll
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    if (c0 >= nv) break;                                      // warp-uniform
                    uint32_t v[16];
                    tc_ld_x16(trow + c0, v);
                    tc_wait_ld();
                    const int q = c0 / 32;          // compile-time after unrolling
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int pick = __shfl_sync(0xFFFFFFFFu, BN >= 32 ? pp[q] : pp[0], (c0 % 32) + i);
                        if (c0 + i < nv) {
                            ycol[(size_t)pick * a.d] = __uint_as_float(v[i]);
                            chk = fmaf(chk, 0.0f, __uint_as_float(v[i]));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
        }
        if (__any_sync(0xFFFFFFFFu, !isfinite(chk)) && lane == 0) record_error(a.err, MOE_DEV_NAN_SCALE);
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {               // final after the barrier: nothing new is issued past it
        if (warp == 4 && lane == 0) {
            drain_stage_fills(full, NS, issued);
            if (STAGED) drain_stage_fills(satoms, NS, issued);
        }
        if (warp == 5 && lane == 0) tc_drain(drain);
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) record_error(a.err, MOE_DEV_TIMEOUT);
}

// Gate/up for tiles of up to 128 routed rows (large batches), in the
// token-major orientation: D[row, 0..255] = A[row] x [Wg tile; Wu tile]^T,
// M = 128 routed rows, N = 256 (gate features f0..f0+127, then up), K = d.
// The epilogue thread of TMEM lane r holds the 128 gate and 128 up values of
// its row, so h = silu(g) * u and its MXFP4 blocks of 32 features are formed
// in registers, with no shuffles. One accumulator buffer (256 columns). (The
// down GEMM stays weight-major at every batch size: there a warp's 32 lanes
// are 32 consecutive output dims, so its stores of Y are coalesced.)
//
// Scale factors reach TMEM through registers, not tcgen05.cp: the copy that
// replicates a 32-row atom into the four lane quadrants occupies the tensor
// pipe for about half an MMA, and a stage needs six of them for four MMAs.
// Warps 6-9 (one per lane quadrant) instead load each stage's six atoms from
// global memory a few stages ahead and write them with tcgen05.st, which runs
// beside the MMAs; they signal the MMA thread through sfull[stage].
template <int NS>
struct CfgTok {
    // warps 0-3 and 10-13 epilogue (feature blocks 0-1 and 2-3 of their lane quadrant), 4 TMA, 5 MMA,
    // 6-9 scales
    static constexpr int THREADS = 448;
    static constexpr int BLK = 128 * 128;
    static constexpr int A_BYTES = BLK;                 // 128 activation rows x 256 e2m1
    static constexpr int B_BYTES = 2 * BLK;             // gate block, up block (256 rows)
    static constexpr int SF_COLS = 24;                  // activation 8, then per k-group: gate 4 | up 4
    static constexpr int SF_STAGE = 6 * 512;            // staged atoms: activations q0 q1 | gate q0 q1 | up q0 q1
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + NS * A_BYTES;
    static constexpr int OFF_SF = OFF_B + NS * B_BYTES;
    static constexpr int OFF_BAR = OFF_SF + NS * SF_STAGE;
    static constexpr int N_BARS = 4 * NS + 3;           // full, empty, sfull, satoms per stage; accf, acce, drain
    static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static constexpr int TMEM_USED = 256 + SF_COLS * NS;
    static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(TMEM_USED <= 512, "TMEM");
};

template <int NS>
__global__ void __launch_bounds__(448, 1) ffn_gate_up_tokens_kernel(const __grid_constant__ GemmMaps maps,
                                                                    const GemmArgs a) {
    using C = CfgTok<NS>;
    constexpr int BN = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + NS;
    uint64_t* sfull = empty + NS;
    uint64_t* satoms = sfull + NS;      // the stage's scale atoms alone (the writers' wait)
    uint64_t* accf = satoms + NS;
    uint64_t* acce = accf + 1;
    uint64_t* drain = acce + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1); mbar_init(&empty[s], 1); mbar_init(&sfull[s], 4); mbar_init(&satoms[s], 1);
        }
        mbar_init(accf, 1);
        mbar_init(acce, 8);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&maps.b[3]);
    }
    if (warp == 5) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    uint32_t issued = 0;                             // stage fills issued by the producer thread
    pdl_wait();                                      // the work list is the plan kernel's output
    const int n_items = *a.n_work * a.m_tiles;
    const int nc = (a.K + 255) / 256;
    const int atoms = a.K / 128;

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer (one thread)
        if (lane == 0) {
            uint32_t& it = issued;
            bool ok_run = true;
            int4 w_next = blockIdx.x < n_items ? a.work[blockIdx.x / a.m_tiles] : make_int4(0, 0, 0, 0);
            for (int item = blockIdx.x; item < n_items && ok_run; item += gridDim.x) {
                const int4 w = w_next;
                const int nxt = item + gridDim.x;
                if (nxt < n_items) w_next = a.work[nxt / a.m_tiles];
                const int mt = item % a.m_tiles;
                const int slot = w.x, pos0 = w.y;
                const uint8_t* rec = a.arena + (size_t)slot * a.slot_bytes;
                const uint8_t* cg = rec + a.off_codes + (size_t)mt * nc * C::BLK;                  // gate tile
                const uint8_t* cu = rec + a.off_codes + (size_t)(a.F / 128 + mt) * nc * C::BLK;    // up tile
                const uint8_t* sg = rec + a.off_scales + (size_t)mt * atoms * 512;                 // their atoms
                const uint8_t* su = rec + a.off_scales + (size_t)(a.F / 128 + mt) * atoms * 512;
                const uint8_t* sa = a.b_scales + (size_t)(pos0 / BN) * atoms * 512;                // activations'
                for (int kc = 0; kc < nc; ++kc, ++it) {
                    const int s = (int)(it % NS);
                    const uint32_t r = it / NS;
                    if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, a.wait_ns)) { ok_run = false; break; }
                    uint8_t* As = smem + C::OFF_A + s * C::A_BYTES;
                    uint8_t* Bs = smem + C::OFF_B + s * C::B_BYTES;
                    uint8_t* Ss = smem + C::OFF_SF + s * C::SF_STAGE;
                    const int at0 = 2 * kc;
                    const uint32_t sf_bytes = (uint32_t)(atoms - at0 < 2 ? atoms - at0 : 2) * 512u;
                    // the scale atoms first, on their own barrier: the writers move them into TMEM while
                    // the operands are still arriving
                    mbar_arrive_expect_tx(&satoms[s], 3 * sf_bytes);
                    bulk_load(Ss, sa + (size_t)at0 * 512, sf_bytes, &satoms[s]);
                    bulk_load(Ss + 1024, sg + (size_t)at0 * 512, sf_bytes, &satoms[s]);
                    bulk_load(Ss + 2048, su + (size_t)at0 * 512, sf_bytes, &satoms[s]);
                    mbar_arrive_expect_tx(&full[s], C::A_BYTES + C::B_BYTES);
                    tma_load_2d(As, &maps.b[3], &full[s], kc * 128, pos0);
                    bulk_load(Bs, cg + (size_t)kc * C::BLK, C::BLK, &full[s]);
                    bulk_load(Bs + C::BLK, cu + (size_t)kc * C::BLK, C::BLK, &full[s]);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // the same lean feed loop as the weight-major kernel's
            int s = 0;
            uint32_t ph = 0, j = 0;
            bool ok_run = true;
            const uint64_t a_base = smem_desc_sw128(smem_u32(smem + C::OFF_A));
            const uint64_t b_base = smem_desc_sw128(smem_u32(smem + C::OFF_B));
            constexpr uint32_t id0 = idesc_mxf4(256, 0, 0), id1 = idesc_mxf4(256, 2, 2);
            for (int item = blockIdx.x; item < n_items && ok_run; item += gridDim.x, ++j) {
                if (!mbar_wait(acce, (j & 1) ^ 1, abort_flag, a.wait_ns)) break;
                tc_fence_after();
                for (int kc = 0; kc < nc; ++kc) {
                    if (!mbar_wait(&full[s], ph, abort_flag, a.wait_ns) || !mbar_wait(&sfull[s], ph, abort_flag, a.wait_ns)) {
                        ok_run = false;
                        break;
                    }
                    tc_fence_after();
                    const int rem = (a.K - kc * 256) / 64;
                    const uint32_t sfc = tmem + 256 + s * C::SF_COLS;
                    const uint64_t ad = a_base + (uint32_t)(s * C::A_BYTES >> 4);
                    const uint64_t bd = b_base + (uint32_t)(s * C::B_BYTES >> 4);
                    const uint32_t acc0 = kc != 0 ? 1u : 0u;
                    if (rem >= 4) {
                        tc_mma_mxf4(tmem, ad, bd, id0, sfc, sfc + 8, acc0);
                        tc_mma_mxf4(tmem, ad + 2, bd + 2, id1, sfc, sfc + 8, 1u);
                        tc_mma_mxf4(tmem, ad + 4, bd + 4, id0, sfc + 4, sfc + 16, 1u);
                        tc_mma_mxf4(tmem, ad + 6, bd + 6, id1, sfc + 4, sfc + 16, 1u);
                    } else {
                        for (int kk = 0; kk < rem; ++kk)
                            tc_mma_mxf4(tmem, ad + 2 * kk, bd + 2 * kk, (kk & 1) ? id1 : id0, sfc + (kk >> 1) * 4,
                                        sfc + 8 + (kk >> 1) * 8, (kc | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);
                    if (++s == NS) { s = 0; ph ^= 1; }
                }
                if (ok_run) tc_commit(accf);
            }
        }
    } else if (warp >= 6 && warp < 10) {
        // ------------------------------------------------------------ scale factors -> TMEM
        // stage g of this CTA is K chunk g % nc of its item g / nc; TMEM column order: activations
        // q = 0, 1, then (gate, up) per q; staged in shared memory as activations q0 q1 | gate q0 q1 |
        // up q0 q1 (one bulk copy per matrix)
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        auto valid = [&](int g) {
            const int at0 = 2 * (g % nc);
            return atoms - at0 < 2 ? atoms - at0 : 2;
        };
        auto slot_of_atom = [](int q, int nvalid) {
            const int kq = q < 2 ? q : (q - 2) >> 1;            // k-group of this column pair
            if (kq >= nvalid) return -1;
            return q < 2 ? q : (((q - 2) & 1) == 0 ? 2 + kq : 4 + kq);
        };
        scale_writer_smem<6, NS>(my_items * nc, valid, slot_of_atom, satoms, sfull, smem + C::OFF_SF, C::SF_STAGE,
                                 tmem + ((uint32_t)((warp & 3) * 32) << 16) + 256, C::SF_COLS, abort_flag,
                                 a.wait_ns);
    } else {
        // ------------------------------------------------------------ epilogue: lane = routed row
        float chk = 0.0f;                                // sticky non-finite detector, as in the kernel above
        uint32_t j = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
            const int4 w = a.work[item / a.m_tiles];
            const int mt = item % a.m_tiles;
            const int pos0 = w.y, nv = w.z;
            if (!warp_wait(accf, j & 1, abort_flag, a.wait_ns)) break;
            tc_fence_after();
            const int quad = warp & 3;                              // TMEM lane quadrant of this warp
            const int row = quad * 32 + lane;
            const int pos = pos0 + row;
            const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
            const int fb0 = warp < 4 ? 0 : 2;
            // 2 of the 4 blocks of 32 features: the raw gate and up values of both are read
            // from TMEM (eight loads in flight at once) and the accumulator is released to the
            // next item's MMAs before any SwiGLU: its two MUFU operations per value would
            // otherwise hold the accumulator for ~2,000 cycles per tile
            uint32_t r[8][16];                  // block q2: gate lo, gate hi, up lo, up hi at 4 q2 ..
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int fb = fb0 + q2;
                tc_ld_x16(trow + 32 * fb, r[4 * q2 + 0]);
                tc_ld_x16(trow + 32 * fb + 16, r[4 * q2 + 1]);
                tc_ld_x16(trow + 128 + 32 * fb, r[4 * q2 + 2]);
                tc_ld_x16(trow + 128 + 32 * fb + 16, r[4 * q2 + 3]);
            }
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce);
            float h[2][32];
            float amax[2] = {0.0f, 0.0f};
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    h[q2][i] = silu_mul(__uint_as_float(r[4 * q2 + (i >> 4)][i & 15]),
                                        __uint_as_float(r[4 * q2 + 2 + (i >> 4)][i & 15]));
                    amax[q2] = fmaxf(amax[q2], fabsf(h[q2][i]));
                }
            if (row < nv) {
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
                    for (int i = 0; i < 32; ++i) chk = fmaf(chk, 0.0f, h[q2][i]);
            }
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int X = mx_shared_exp(amax[q2]);
                const float inv = exp2_int(-X);
                uint32_t wd[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) wd[q] = e2m1x8(h[q2] + q * 8, inv);
                if (row < nv) {
                    const int f = mt * 128 + 32 * (fb0 + q2);
                    *reinterpret_cast<uint4*>(a.hq + (size_t)pos * (a.F / 2) + f / 2) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    a.hsp[operand_scale_offset(pos, f / 32, BN, a.F)] = (uint8_t)(X + 127);
                }
            }
        }
        if (__any_sync(0xFFFFFFFFu, !isfinite(chk)) && lane == 0) record_error(a.err, MOE_DEV_NAN_SCALE);
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {               // final after the barrier: nothing new is issued past it
        if (warp == 4 && lane == 0) { drain_stage_fills(full, NS, issued); drain_stage_fills(satoms, NS, issued); }
        if (warp == 5 && lane == 0) tc_drain(drain);
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) record_error(a.err, MOE_DEV_TIMEOUT);
}

// A CTA shaped like the pipelines above (TMEM allocated by warp 5, an MMA
// thread that has committed work, warps waiting on an mbarrier) whose wait can
// never be satisfied: nothing arrives on `never`. Every wait gives up after
// the bound in force and the CTA takes the same exit as a stalled pipeline
// (drain, free TMEM, MOE_DEV_TIMEOUT), so a caller can check that a stall ends
// in an error status instead of a hang.
__global__ void __launch_bounds__(128, 1) wait_selftest(uint32_t* err, uint64_t wait_ns) {
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_word;
    uint64_t* never = &bars[0];
    uint64_t* drain = &bars[1];
    volatile int* abort_flag = &abort_word;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    if (threadIdx.x == 0) {
        mbar_init(never, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc(&tmem_slot, 32); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    const uint32_t tmem = tmem_slot;
    (void)warp_wait(never, 0, abort_flag, wait_ns);
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (warp == 1 && lane == 0) tc_drain(drain);
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
    if (threadIdx.x == 0 && *abort_flag) record_error(err, MOE_DEV_TIMEOUT);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

cudaError_t encode(CUtensorMap* m, const uint8_t* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<uint8_t*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Activation operand rows: (row bytes, positions); boxes of 16, 32, 64 and 128 rows.
cudaError_t make_act_maps(CUtensorMap* m, const uint8_t* base, uint64_t row_bytes, uint64_t rows) {
    for (int i = 0; i < 4; ++i) {
        cuuint64_t dims[2] = {row_bytes, rows};
        cuuint64_t strides[1] = {row_bytes};
        cuuint32_t box[2] = {128, (cuuint32_t)(16 << i)};
        cudaError_t e = encode(&m[i], base, 2, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int MODE, int BN, int NS, int KCH, int NBUF, bool STAGED = false>
cudaError_t launch_one(const GemmMaps& maps, const GemmArgs& g, long max_items, cudaStream_t s) {
    using C = Cfg<MODE, BN, NS, KCH, NBUF, STAGED>;
    auto kern = ffn_gemm_kernel<MODE, BN, NS, KCH, NBUF, STAGED>;
    static int occ_cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int occ = dev < 64 ? occ_cache[dev] : 0;
    if (occ == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::THREADS, C::SMEM);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        const int tmem_fit = 512 / C::TMEM_COLS;
        if (occ > tmem_fit) occ = tmem_fit;
        if (dev < 64) occ_cache[dev] = occ;
    }
    if (max_items <= 0) return cudaSuccess;
    long grid = (long)occ * moe_sm_count();
    if (grid > max_items) grid = max_items;
    moe_prof_begin(MODE == 1 ? MK_GEMM_GATE_UP : MK_GEMM_DOWN, s);
    const cudaError_t e = moe_launch(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, s, maps, g);
    moe_prof_end(MODE == 1 ? MK_GEMM_GATE_UP : MK_GEMM_DOWN, s);
    moe_count_launches(1);
    return e;
}

template <int NS>
cudaError_t launch_tokens(const GemmMaps& maps, const GemmArgs& g, long max_items, cudaStream_t s) {
    using C = CfgTok<NS>;
    auto kern = ffn_gate_up_tokens_kernel<NS>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    if (max_items <= 0) return cudaSuccess;
    long grid = moe_sm_count();                    // one CTA per SM (TMEM: 512 columns each)
    if (grid > max_items) grid = max_items;
    moe_prof_begin(MK_GEMM_GATE_UP, s);
    const cudaError_t e = moe_launch(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, s, maps, g);
    moe_prof_end(MK_GEMM_GATE_UP, s);
    moe_count_launches(1);
    return e;
}

template <int MODE>
cudaError_t launch_mode(const GemmMaps& maps, const GemmArgs& g, long max_items, int bn, cudaStream_t s) {
    // Scale atoms staged in shared memory (STAGED) where the stages leave room and it measured
    // faster: the 16-row gate/up tiles (one token: 53.5 -> 51 us per layer step) and the
    // token-major gate/up kernel; the 64-row and down tiles were no faster staged.
    // 64 KB of weights per stage: with fewer CTAs streaming than SMs, one SM takes about
    // 100 GB/s from HBM through five 32 KB stages and 140-160 GB/s through three 64 KB ones
    // (measured with a per-SM bulk-copy streaming test), which is what the CTAs left in a
    // partial last round, or in a grid of few items, get.
    if constexpr (MODE == 1) {   // gate + up tiles, two 256-element K chunks per stage
        switch (bn) {
            case 16: return launch_one<MODE, 16, 3, 2, 2, true>(maps, g, max_items, s);    // atoms staged
            case 32: return launch_one<MODE, 32, 3, 2, 2>(maps, g, max_items, s);
            case 64: return launch_one<MODE, 64, 2, 2, 2>(maps, g, max_items, s);
            default: return launch_one<MODE, 128, 4, 1, 1>(maps, g, max_items, s);
        }
    }
    else switch (bn) {      // one tile, four chunks per stage
        case 16: return launch_one<MODE, 16, 3, 4, 2>(maps, g, max_items, s);
        case 32: return launch_one<MODE, 32, 2, 4, 2>(maps, g, max_items, s);
        case 64: return launch_one<MODE, 64, 2, 4, 2>(maps, g, max_items, s);
        default: return launch_one<MODE, 128, 3, 2, 2>(maps, g, max_items, s);
    }
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t wait_ns, cudaStream_t s) {
    moe_count_launches(1);
    return moe_launch(wait_selftest, dim3(1), dim3(128), 0, s, err, wait_ns);
}

cudaError_t launch_ffn_gemms(const FfnLaunch& a, cudaStream_t s, int* n_launches) {
    const moe_arena& ar = *a.arena;
    const uint8_t* base = static_cast<const uint8_t*>(ar.base);
    GemmMaps m1, m2;
    cudaError_t e = make_act_maps(m1.b, a.xp, (uint64_t)a.d / 2, (uint64_t)a.pad_max);
    if (e == cudaSuccess) e = make_act_maps(m2.b, a.hq, (uint64_t)a.F / 2, (uint64_t)a.pad_max);
    if (e != cudaSuccess) return e;

    GemmArgs g{};
    g.arena = base;
    g.slot_bytes = ar.slot_bytes;
    g.F = a.F;
    g.d = a.d;
    g.work = a.work;
    g.n_work = a.n_work;
    g.pair_of_pos = a.pair_of_pos;
    g.err = a.err;
    g.wait_ns = a.wait_ns;
    // Decode tiles (up to 64 rows) read each weight tile once per call: streamed evict-first so that
    // the 100-200 MB of weights a decode layer reads do not push the following small kernels' code and
    // data (routing tables, logits, activations) out of L2. Large batches reuse each weight tile
    // across their token tiles and keep the default policy.
    g.evict_first = a.bn <= 64 ? 1 : 0;

    GemmArgs g1 = g;       // gate/up + SwiGLU
    g1.off_codes = ar.off_gu_codes;
    g1.off_scales = ar.off_gu_scales;
    g1.K = a.d;
    g1.m_tiles = a.F / 128;
    g1.b_scales = a.xsp;
    g1.hq = a.hq;
    g1.hsp = a.hsp;
    if (a.bn == 128) e = launch_tokens<4>(m1, g1, (long)a.work_max * g1.m_tiles, s);   // large batches
    else e = launch_mode<1>(m1, g1, (long)a.work_max * g1.m_tiles, a.bn, s);
    if (e != cudaSuccess) return e;

    GemmArgs g2 = g;       // down
    g2.off_codes = ar.off_dn_codes;
    g2.off_scales = ar.off_dn_scales;
    g2.K = a.F;
    g2.m_tiles = a.d / 128;
    g2.b_scales = a.hsp;
    g2.Y = a.Y;

    e = launch_mode<2>(m2, g2, (long)a.work_max * g2.m_tiles, a.bn, s);
    if (n_launches) *n_launches = 2;
    return e;
}
