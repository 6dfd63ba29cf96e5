// ttt_mlp_w8.cuh -- body of the eight-warp TTT-MLP kernel (d = 64, m = 256, mini-batches
// of at most 16 tokens), included by ttt_mlp_bf16.cu twice: W8_LN 0 gives the plain inner
// model act(x W1 + c1) W2 + c2, W8_LN 1 the inner norm and residual x + LN(...) of the
// walkthrough's TTT-MLP (section 2.2.1): the residual of a key is the layer-norm backward
// of f(k) - v, and z = q + LN(y_q), each token's statistics over its 64 outputs summed
// across the four warps that hold them (quad shuffle, then a shared-memory exchange at a
// named barrier).  W8_KERNEL names the kernel, W8_CFG its shared-memory layout and
// W8_PARAMS its parameters.
template <int ACT>
__global__ void __launch_bounds__(W8_CFG::THREADS, 1)
    W8_KERNEL(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const W8_PARAMS p)
{
    using C = W8_CFG;
    constexpr int D = C::D, M = C::M, NK = C::NK, NKM = C::NKM, NJ = C::NJ, NS = C::NS, NW = C::NW;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x, T = p.T;
    const int g = lane >> 2, t4 = lane & 3;
    const int rowA = (lane & 7) + 8 * ((lane >> 3) & 1), colA = 8 * (lane >> 4);
    const int rowB = (lane & 7) + 8 * (lane >> 4), colB = 8 * ((lane >> 3) & 1);
    const bool has_eta = p.eta != nullptr;
    const uint32_t bar_full = base + C::BAR_OFF;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::BAR_OFF + NS * 8);
    const uint32_t AK = base + C::AK_OFF, AQ = base + C::AQ_OFF;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar_full + 8 * s, 1 + (has_eta ? 32 : 0));
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ---------------------------------------------------------- initial state
    const int w = warp;
    const size_t ps = p.per_batch ? (size_t)bh : (size_t)(bh % p.H);
    const float *W1g = p.W1 + ps * D * M, *c1g = p.c1 + ps * M;
    const float *W2g = p.W2 + ps * M * D, *c2g = p.c2 + ps * D;
    // group hg (hidden 32w + 16hg ..): w1[hg][j] = W1^T rows (+g, +g+8) x columns 8j + 2t4 .. +1
    float w1[2][NJ][4];
    // w2[hg][mt][nt] = W2[h + 2t4 .. +1][16mt + g (+8)], h = 32w + 16hg + 8nt
    float w2[2][NK][2][4];
    float c1r[2][2][2];  // c1 of hidden 32w + 16hg + 8nt + 2t4 + i
#pragma unroll
    for (int hg = 0; hg < 2; ++hg) {
        const int h0 = 32 * w + 16 * hg;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int r = 8 * j + 2 * t4;
            w1[hg][j][0] = W1g[(size_t)r * M + h0 + g];
            w1[hg][j][1] = W1g[(size_t)(r + 1) * M + h0 + g];
            w1[hg][j][2] = W1g[(size_t)r * M + h0 + g + 8];
            w1[hg][j][3] = W1g[(size_t)(r + 1) * M + h0 + g + 8];
        }
#pragma unroll
        for (int mt = 0; mt < NK; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int hr = h0 + 8 * nt + 2 * t4, dc = 16 * mt + g;
                w2[hg][mt][nt][0] = W2g[(size_t)hr * D + dc];
                w2[hg][mt][nt][1] = W2g[(size_t)(hr + 1) * D + dc];
                w2[hg][mt][nt][2] = W2g[(size_t)hr * D + dc + 8];
                w2[hg][mt][nt][3] = W2g[(size_t)(hr + 1) * D + dc + 8];
            }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 2; ++i) c1r[hg][nt][i] = c1g[h0 + 8 * nt + 2 * t4 + i];
    }
    // c2 of columns 16w + 8nt + 2t4 + i (kept by warps 0-3, which form E)
    float c2r[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 2; ++i) c2r[nt][i] = w < 4 ? c2g[16 * w + 8 * nt + 2 * t4 + i] : 0.f;
    // bf16 copy of this warp's W2 rows into buffer `buf` ([hidden][d], transposed
    // stores of the accumulator tiles)
    auto put_w2 = [&](uint32_t buf) {
        const int blk = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int hg = 0; hg < 2; ++hg)
#pragma unroll
            for (int mt = 0; mt < NK; ++mt)
                stsm_x4_t(buf + (uint32_t)(32 * w + 16 * hg + 8 * (blk >> 1) + rr) * C::W2R +
                              (uint32_t)(16 * mt + 8 * (blk & 1)) * 2,
                          pack_bf16(w2[hg][mt][0][0], w2[hg][mt][0][1]),
                          pack_bf16(w2[hg][mt][0][2], w2[hg][mt][0][3]),
                          pack_bf16(w2[hg][mt][1][0], w2[hg][mt][1][1]),
                          pack_bf16(w2[hg][mt][1][2], w2[hg][mt][1][3]));
    };
    // bf16 W1 of group hg as the B operand of a product with it (k-tile kk):
    // n-tile 0 (hidden +0..7) uses (b[0], b[1]), n-tile 1 (hidden +8..15) (b[2], b[3])
    auto w1_b = [&](int hg, int kk, uint32_t (&b)[4]) {
        b[0] = pack_bf16(w1[hg][2 * kk][0], w1[hg][2 * kk][1]);
        b[1] = pack_bf16(w1[hg][2 * kk + 1][0], w1[hg][2 * kk + 1][1]);
        b[2] = pack_bf16(w1[hg][2 * kk][2], w1[hg][2 * kk][3]);
        b[3] = pack_bf16(w1[hg][2 * kk + 1][2], w1[hg][2 * kk + 1][3]);
    };
    int w2cur = 0;
    put_w2(base + C::W2B_OFF);

    // ------------------------------------------------ token tiles (warp 0 issues)
    JobIter itp(T, p.b, p.causal);
    int issued = 0;
    auto issue_next = [&]() {  // into the stage the chunk NS - 1 back released (after its barrier B3)
        if (!itp.valid()) return;
        const Job J = itp.get();
        const int s = issued % NS;
        const uint32_t st = base + s * C::STAGE, full = bar_full + 8 * s;
        if (has_eta) {
            if (lane < J.c) cp_async_4(st + 3 * C::TILE + 4 * lane, p.eta + (size_t)bh * T + J.t0 + lane);
            cp_async_arrive_noinc(full);
        }
        if (lane == 0) {
            mbar_arrive_expect_tx(full, 3 * C::TILE);
            tma_load_3d(st, &tq, full, 0, J.t0, bh);
            tma_load_3d(st + C::TILE, &tk, full, 0, J.t0, bh);
            tma_load_3d(st + 2 * C::TILE, &tv, full, 0, J.t0, bh);
        }
        __syncwarp();
        itp.next();
        ++issued;
    };
    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tq)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tk)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tv)) : "memory");
        }
        for (int i = 0; i < NS - 1; ++i) issue_next();
    }
    __syncthreads();

    // acc[nt] += X W[:, cc + 8nt .. +7] over all hidden units (X = A_k or A_q,
    // [16][AR] bf16; cc = 16 (w mod 4)); the fragments of the next 32 hidden units
    // load while the current ones multiply
    const int cc = 16 * (w & 3);
    auto col_product16 = [&](uint32_t W, uint32_t X, float (&acc)[2][2][4]) {
        uint32_t fb[2][2][4], fa[2][8];
        auto ld = [&](int kp, int sl) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                ldsm_x4_t(W + (uint32_t)(32 * kp + lane) * C::W2R + (cc + 8 * nt) * 2, fb[sl][nt][0], fb[sl][nt][1],
                          fb[sl][nt][2], fb[sl][nt][3]);
            ldsm_x4(X + rowA * C::AR + (32 * kp + colA) * 2, fa[sl][0], fa[sl][1], fa[sl][2], fa[sl][3]);
            ldsm_x4(X + rowA * C::AR + (32 * kp + 16 + colA) * 2, fa[sl][4], fa[sl][5], fa[sl][6], fa[sl][7]);
        };
        ld(0, 0);
#pragma unroll
        for (int kp = 0; kp < NKM / 2; ++kp) {
            if (kp + 1 < NKM / 2) ld(kp + 1, (kp + 1) & 1);
            const int sl = kp & 1;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                mma_bf16(acc[nt][0], fa[sl][0], fa[sl][1], fa[sl][2], fa[sl][3], fb[sl][nt][0], fb[sl][nt][1]);
                mma_bf16(acc[nt][1], fa[sl][4], fa[sl][5], fa[sl][6], fa[sl][7], fb[sl][nt][2], fb[sl][nt][3]);
            }
        }
    };
    // A_q A_k^T partial sums of all warps -> S2' = M .* (A_q A_k^T + 1) as bf16, one
    // element per thread (c: tokens of that chunk)
    auto reduce_s2 = [&](int c) {
        const int e = 32 * w + lane, r = e >> 4, kc = e & 15;
        const float *sf = reinterpret_cast<const float *>(gbase + C::S2F_OFF);
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < NW; ++u) sum += sf[(u * 16 + r) * C::S2R + kc];
        const bool keep = kc < c && (!p.causal || kc <= r);
        reinterpret_cast<__nv_bfloat16 *>(gbase + C::S2P_OFF + r * 48)[kc] = __float2bfloat16_rn(keep ? sum + 1.f : 0.f);
    };
    // z of a chunk on columns cc .. cc+15: P (its A_q times its W2 copy) + c2 + S2' (-Et),
    // tokens t0 .. t0+c-1; c2 at the chunk's start from the snapshot `c2s`
    auto store_z = [&](const float (&pz)[2][2][4], uint32_t NEBc, int t0, int c, const float *c2s) {
        uint32_t sa[4], b0, b1, b2, b3;
        ldsm_x4(base + C::S2P_OFF + rowA * 48 + colA * 2, sa[0], sa[1], sa[2], sa[3]);
        ldsm_x4_t(NEBc + (uint32_t)(lane & 15) * C::ER + (cc + 8 * (lane >> 4)) * 2, b0, b1, b2, b3);
#if W8_LN
        float zz[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) zz[nt][i] = pz[nt][0][i] + pz[nt][1][i];
            mma_bf16(zz[nt], sa[0], sa[1], sa[2], sa[3], nt ? b2 : b0, nt ? b3 : b1);
            const int col = cc + 8 * nt + 2 * t4;
#pragma unroll
            for (int i = 0; i < 4; ++i) zz[nt][i] += c2s[col + (i & 1)];
        }
        {  // z = q + LN(y_q), statistics over the 64 outputs of each query
            float s1[2] = {}, s2[2] = {};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    s1[i >> 1] += zz[nt][i];
                    s2[i >> 1] += zz[nt][i] * zz[nt][i];
                }
            w8_row_sums(s1, s2, reinterpret_cast<float2 *>(gbase + C::LNR_OFF) + 2 * 64, w & 3, g, t4, 2);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float mu = s1[r] * (1.f / D);
                const float rs = rsqrtf(fmaxf(s2[r] * (1.f / D) - mu * mu, 0.f) + p.ln_eps);
                const int tok = g + 8 * r;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = cc + 8 * nt + 2 * t4;
                    const float *gh = p.ln_gamma + (size_t)(bh % p.H) * D + col, *bt = p.ln_beta + (size_t)(bh % p.H) * D + col;
                    const float lg[2][2] = {{gh[0], gh[1]}, {gh[0], gh[1]}}, lb[2][2] = {{bt[0], bt[1]}, {bt[0], bt[1]}};
                    uint32_t qw = 0;
                    if (tok < c) qw = *reinterpret_cast<const uint32_t *>(p.q + ((size_t)bh * T + t0 + tok) * D + col);
                    zz[nt][2 * r] = bf16_lo(qw) + lg[nt][0] * (zz[nt][2 * r] - mu) * rs + lb[nt][0];
                    zz[nt][2 * r + 1] = bf16_hi(qw) + lg[nt][1] * (zz[nt][2 * r + 1] - mu) * rs + lb[nt][1];
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = cc + 8 * nt + 2 * t4;
            __nv_bfloat16 *zb = p.z + ((size_t)bh * T + t0) * D + col;
            if (g < c) *reinterpret_cast<uint32_t *>(zb + (size_t)g * D) = pack_bf16(zz[nt][0], zz[nt][1]);
            if (g + 8 < c) *reinterpret_cast<uint32_t *>(zb + (size_t)(g + 8) * D) = pack_bf16(zz[nt][2], zz[nt][3]);
        }
#else
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float zz[4] = {pz[nt][0][0] + pz[nt][1][0], pz[nt][0][1] + pz[nt][1][1], pz[nt][0][2] + pz[nt][1][2],
                           pz[nt][0][3] + pz[nt][1][3]};
            mma_bf16(zz, sa[0], sa[1], sa[2], sa[3], nt ? b2 : b0, nt ? b3 : b1);
            const int col = cc + 8 * nt + 2 * t4;
            const float x = c2s[col], y = c2s[col + 1];
            __nv_bfloat16 *zb = p.z + ((size_t)bh * T + t0) * D + col;
            if (g < c) *reinterpret_cast<uint32_t *>(zb + (size_t)g * D) = pack_bf16(zz[0] + x, zz[1] + y);
            if (g + 8 < c) *reinterpret_cast<uint32_t *>(zb + (size_t)(g + 8) * D) = pack_bf16(zz[2] + x, zz[3] + y);
        }
#endif
    };
    int prev_t0 = 0, prev_c = 0;   // the previous chunk, whose outputs are finished one chunk later

    // ---------------------------------------------------------------- chunks
    JobIter it(T, p.b, p.causal);
    int jb = 0;
    for (; it.valid(); it.next(), ++jb) {
        const Job J = it.get();
        if (warp == 0) issue_next();
        const int s = jb % NS;
        const uint32_t tQ = base + s * C::STAGE, tK = tQ + C::TILE, tV = tQ + 2 * C::TILE;
        const float *eta_s = reinterpret_cast<const float *>(gbase + s * C::STAGE + 3 * C::TILE);
        auto eta_of = [&](int tok) -> float { return has_eta ? eta_s[tok] : p.eta_scalar; };
        // bf16 W2 at this mini-batch's start; the other buffer holds the previous
        // chunk's copy (its queries are finished in phase 2) and then receives the next
        const uint32_t W2B = base + C::W2B_OFF + (uint32_t)(w2cur * M * C::W2R);
        const uint32_t W2N = base + C::W2B_OFF + (uint32_t)((w2cur ^ 1) * M * C::W2R);
        const uint32_t EB = base + C::EB_OFF + (uint32_t)((jb & 1) * 16 * C::ER);
        const uint32_t NEB = base + C::NEB_OFF + (uint32_t)((jb & 1) * 16 * C::ER);
        const uint32_t NEBp = base + C::NEB_OFF + (uint32_t)(((jb & 1) ^ 1) * 16 * C::ER);
        if (!mbar_wait(bar_full + 8 * s, (jb / NS) & 1, p.status, kSiteConsumerFull)) *abort_flag = 1;

        // phase 1: H_k = K W1 + c1, A_k = SiLU(H_k), SiLU'(H_k); scores for the queries
        uint32_t kf[NK][4];
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) ldsm_x4(tK + mtoff<D>(rowA, 16 * kk + colA), kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3]);
        float sp[2][2][4];
        uint32_t akp[2][4];
#pragma unroll
        for (int hg = 0; hg < 2; ++hg) {
            float hk[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t b[4];
                w1_b(hg, kk, b);
                mma_bf16(hk[0], kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3], b[0], b[1]);
                mma_bf16(hk[1], kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3], b[2], b[3]);
            }
            float ak[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    act_d<ACT>(hk[nt][i] + c1r[hg][nt][i & 1], ak[nt][i], sp[hg][nt][i]);
                }
            akp[hg][0] = pack_bf16(ak[0][0], ak[0][1]);  // (tok 0-7, hidden 0-7 of the group)
            akp[hg][1] = pack_bf16(ak[0][2], ak[0][3]);  // (tok 8-15, hidden 0-7)
            akp[hg][2] = pack_bf16(ak[1][0], ak[1][1]);  // (tok 0-7, hidden 8-15)
            akp[hg][3] = pack_bf16(ak[1][2], ak[1][3]);  // (tok 8-15, hidden 8-15)
            stsm_x4(AK + rowA * C::AR + (32 * w + 16 * hg + colA) * 2, akp[hg][0], akp[hg][1], akp[hg][2],
                    akp[hg][3]);
        }
        if (w >= NW - 2) {
            // S' = M .* (Q K^T + 1): warp NW-2 forms keys 0-7, warp NW-1 keys 8-15
            const int nt = w - (NW - 2);
            uint32_t qa[NK][4];
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) ldsm_x4(tQ + mtoff<D>(rowA, 16 * kk + colA), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            // K's A fragments are the B operand: keys 8nt + g take registers nt, nt + 2
            float sc[4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk)
                mma_bf16(sc, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], nt ? kf[kk][1] : kf[kk][0], nt ? kf[kk][3] : kf[kk][2]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tq_ = g + 8 * (i >> 1), ss = 8 * nt + 2 * t4 + (i & 1);
                const bool keep = ss < J.c && (!p.causal || ss <= tq_);
                sc[i] = keep ? sc[i] + 1.f : 0.f;
            }
            const uint32_t addr = base + C::SP_OFF + (uint32_t)((lane & 7) + 8 * ((lane >> 3) & 1)) * 48 + 16 * nt;
            asm volatile("stmatrix.sync.aligned.m8n8.x2.shared.b16 [%0], {%1,%2};" ::"r"(addr),
                         "r"(pack_bf16(sc[0], sc[1])), "r"(pack_bf16(sc[2], sc[3]))
                         : "memory");
        }
        if (jb > 0) reduce_s2(prev_c);  // the previous chunk's partials (written before its B3)
        __syncthreads();  // B1: A_k, S', previous S2' visible
        if (*abort_flag) break;

        // phase 2: warps 0-3: E = A_k W2 + c2 - V and -Et on columns 16w .. 16w+15;
        // warps 4-7: the previous chunk's P = A_q W2 and z on columns 16(w-4) ..
        float cs2[2][2] = {};  // column sums of -Et (the c2 write of this mini-batch)
        if (w < 4) {
            float e[2][2][4] = {};
            col_product16(W2B, AK, e);
            float *c2snap = reinterpret_cast<float *>(gbase + C::C2S_OFF) + (jb & 1) * D;
#if W8_LN
            // LN: the residual of key t is the layer-norm backward of f(k_t) - v_t,
            // (gamma / sigma) (g - mean(g) - xhat mean(g xhat)), g = gamma (k + LN(y) - v)
            float lnr[2][2][2];  // [nt][row][i]
            {
                float lg[2][2], lb[2][2];  // scale / shift of columns cc + 8 nt + 2 t4 + i
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        lg[nt][i] = p.ln_gamma[(size_t)(bh % p.H) * D + cc + 8 * nt + 2 * t4 + i];
                        lb[nt][i] = p.ln_beta[(size_t)(bh % p.H) * D + cc + 8 * nt + 2 * t4 + i];
                    }
                float y[2][2][2], s1[2] = {}, s2[2] = {};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            y[nt][r][i] = e[nt][0][2 * r + i] + e[nt][1][2 * r + i] + c2r[nt][i];
                            s1[r] += y[nt][r][i];
                            s2[r] += y[nt][r][i] * y[nt][r][i];
                        }
                w8_row_sums(s1, s2, reinterpret_cast<float2 *>(gbase + C::LNR_OFF), w & 3, g, t4, 1);
                float rs[2], g1[2] = {}, g2[2] = {}, gv[2][2][2], xh[2][2][2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float mu = s1[r] * (1.f / D);
                    rs[r] = rsqrtf(fmaxf(s2[r] * (1.f / D) - mu * mu, 0.f) + p.ln_eps);
                    const int tok = g + 8 * r;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int col = cc + 8 * nt + 2 * t4;
                        const uint32_t kw = *reinterpret_cast<const uint32_t *>(gbase + (tK - base) + mtoff<D>(tok, col));
                        const uint32_t vw = *reinterpret_cast<const uint32_t *>(gbase + (tV - base) + mtoff<D>(tok, col));
                        const float kv[2] = {bf16_lo(kw), bf16_hi(kw)}, vv[2] = {bf16_lo(vw), bf16_hi(vw)};
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            xh[nt][r][i] = (y[nt][r][i] - mu) * rs[r];
                            gv[nt][r][i] = lg[nt][i] * (kv[i] + lg[nt][i] * xh[nt][r][i] + lb[nt][i] - vv[i]);
                            g1[r] += gv[nt][r][i];
                            g2[r] += gv[nt][r][i] * xh[nt][r][i];
                        }
                    }
                }
                w8_row_sums(g1, g2, reinterpret_cast<float2 *>(gbase + C::LNR_OFF) + 64, w & 3, g, t4, 1);
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            lnr[nt][r][i] = rs[r] * (gv[nt][r][i] - g1[r] * (1.f / D) - xh[nt][r][i] * g2[r] * (1.f / D));
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = cc + 8 * nt + 2 * t4;
                if (g == 0) {
                    c2snap[col] = c2r[nt][0];
                    c2snap[col + 1] = c2r[nt][1];
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {  // token rows g, g + 8
                    const int tok = g + 8 * r;
                    const float ex = lnr[nt][r][0];
                    const float ey = lnr[nt][r][1];
                    const bool ok = tok < J.c;
                    const float et = -eta_of(tok);
                    const float nx = ok ? et * ex : 0.f, ny = ok ? et * ey : 0.f;
                    cs2[nt][0] += nx;
                    cs2[nt][1] += ny;
                    *reinterpret_cast<uint32_t *>(gbase + (EB - base) + tok * C::ER + col * 2) = pack_bf16(ex, ey);
                    *reinterpret_cast<uint32_t *>(gbase + (NEB - base) + tok * C::ER + col * 2) = pack_bf16(nx, ny);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    cs2[nt][i] += __shfl_xor_sync(0xffffffffu, cs2[nt][i], 4);
                    cs2[nt][i] += __shfl_xor_sync(0xffffffffu, cs2[nt][i], 8);
                    cs2[nt][i] += __shfl_xor_sync(0xffffffffu, cs2[nt][i], 16);
                }
            }
#else
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = cc + 8 * nt + 2 * t4;
                if (g == 0) {
                    c2snap[col] = c2r[nt][0];
                    c2snap[col + 1] = c2r[nt][1];
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {  // token rows g, g + 8
                    const int tok = g + 8 * r;
                    const uint32_t vw = *reinterpret_cast<const uint32_t *>(gbase + (tV - base) + mtoff<D>(tok, col));
                    const float ex = e[nt][0][2 * r] + e[nt][1][2 * r] + c2r[nt][0] - bf16_lo(vw);
                    const float ey = e[nt][0][2 * r + 1] + e[nt][1][2 * r + 1] + c2r[nt][1] - bf16_hi(vw);
                    const bool ok = tok < J.c;
                    const float et = -eta_of(tok);
                    const float nx = ok ? et * ex : 0.f, ny = ok ? et * ey : 0.f;
                    cs2[nt][0] += nx;
                    cs2[nt][1] += ny;
                    *reinterpret_cast<uint32_t *>(gbase + (EB - base) + tok * C::ER + col * 2) = pack_bf16(ex, ey);
                    *reinterpret_cast<uint32_t *>(gbase + (NEB - base) + tok * C::ER + col * 2) = pack_bf16(nx, ny);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    cs2[nt][i] += __shfl_xor_sync(0xffffffffu, cs2[nt][i], 4);
                    cs2[nt][i] += __shfl_xor_sync(0xffffffffu, cs2[nt][i], 8);
                    cs2[nt][i] += __shfl_xor_sync(0xffffffffu, cs2[nt][i], 16);
                }
            }
#endif
        } else if (jb > 0) {
            float pz[2][2][4] = {};
            col_product16(W2N, AQ, pz);
            store_z(pz, NEBp, prev_t0, prev_c, reinterpret_cast<const float *>(gbase + C::C2S_OFF) + ((jb - 1) & 1) * D);
        }
        __syncthreads();  // B2: E, -Et visible; the previous chunk's A_q and W2 copy no longer read

        // phase 3: delta; query pre-activations (W1, c1 of the mini-batch start);
        // then the weight updates and the next bf16 W2 copy
        uint32_t ef[NK][4];
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) ldsm_x4(EB + rowA * C::ER + (16 * kk + colA) * 2, ef[kk][0], ef[kk][1], ef[kk][2], ef[kk][3]);
        uint32_t dfr[2][4];  // -Dt^T blocks per group: (h 0-7, tok 0-7), (h 8-15, tok 0-7), (h 0-7, tok 8-15), (h 8-15, tok 8-15)
        float cs1[2][2][2] = {};  // column sums of -Dt (the c1 write)
#pragma unroll
        for (int hg = 0; hg < 2; ++hg) {
            float dl[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(W2B + (uint32_t)(32 * w + 16 * hg + rowB) * C::W2R + (16 * kk + colB) * 2, b0, b1, b2, b3);
                mma_bf16(dl[0], ef[kk][0], ef[kk][1], ef[kk][2], ef[kk][3], b0, b1);
                mma_bf16(dl[1], ef[kk][0], ef[kk][1], ef[kk][2], ef[kk][3], b2, b3);
            }
            float nd[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = g + 8 * (i >> 1);
                    nd[nt][i] = tok < J.c ? -eta_of(tok) * dl[nt][i] * sp[hg][nt][i] : 0.f;
                    cs1[hg][nt][i & 1] += nd[nt][i];
                }
            dfr[hg][0] = movmatrix_t(pack_bf16(nd[0][0], nd[0][1]));
            dfr[hg][1] = movmatrix_t(pack_bf16(nd[1][0], nd[1][1]));
            dfr[hg][2] = movmatrix_t(pack_bf16(nd[0][2], nd[0][3]));
            dfr[hg][3] = movmatrix_t(pack_bf16(nd[1][2], nd[1][3]));
        }
        float aq[2][2][4];
        {
            uint32_t qf[NK][4], spf[4];
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) ldsm_x4(tQ + mtoff<D>(rowA, 16 * kk + colA), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
            ldsm_x4(base + C::SP_OFF + rowA * 48 + colA * 2, spf[0], spf[1], spf[2], spf[3]);
#pragma unroll
            for (int hg = 0; hg < 2; ++hg) {
                // H_q = Q W1 + c1 + S' (-Dt); A_q = SiLU(H_q) -> shared
                float hq[2][4] = {};
#pragma unroll
                for (int kk = 0; kk < NK; ++kk) {
                    uint32_t b[4];
                    w1_b(hg, kk, b);
                    mma_bf16(hq[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b[0], b[1]);
                    mma_bf16(hq[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b[2], b[3]);
                }
                mma_bf16(hq[0], spf[0], spf[1], spf[2], spf[3], dfr[hg][0], dfr[hg][2]);
                mma_bf16(hq[1], spf[0], spf[1], spf[2], spf[3], dfr[hg][1], dfr[hg][3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        aq[hg][nt][i] = act<ACT>(hq[nt][i] + c1r[hg][nt][i & 1]);
                    }
                stsm_x4(AQ + rowA * C::AR + (32 * w + 16 * hg + colA) * 2, pack_bf16(aq[hg][0][0], aq[hg][0][1]),
                        pack_bf16(aq[hg][0][2], aq[hg][0][3]), pack_bf16(aq[hg][1][0], aq[hg][1][1]),
                        pack_bf16(aq[hg][1][2], aq[hg][1][3]));
            }
        }
        {
            // W1^T += (-Dt^T) K,  W2 += A_k^T (-Et) (as W2^T += (-Et^T) A_k tiles)
            uint32_t ktf[NK][4], nef[NK][4];
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                ldsm_x4_t(tK + mtoff<D>(rowA, 16 * kk + colA), ktf[kk][0], ktf[kk][1], ktf[kk][2], ktf[kk][3]);
                ldsm_x4_t(NEB + rowB * C::ER + (16 * kk + colB) * 2, nef[kk][0], nef[kk][1], nef[kk][2], nef[kk][3]);
            }
#pragma unroll
            for (int hg = 0; hg < 2; ++hg) {
#pragma unroll
                for (int j2 = 0; j2 < NK; ++j2) {
                    mma_bf16(w1[hg][2 * j2], dfr[hg][0], dfr[hg][1], dfr[hg][2], dfr[hg][3], ktf[j2][0], ktf[j2][1]);
                    mma_bf16(w1[hg][2 * j2 + 1], dfr[hg][0], dfr[hg][1], dfr[hg][2], dfr[hg][3], ktf[j2][2], ktf[j2][3]);
                }
                const uint32_t bt00 = movmatrix_t(akp[hg][0]), bt01 = movmatrix_t(akp[hg][1]);
                const uint32_t bt10 = movmatrix_t(akp[hg][2]), bt11 = movmatrix_t(akp[hg][3]);
#pragma unroll
                for (int mt = 0; mt < NK; ++mt) {
                    mma_bf16(w2[hg][mt][0], nef[mt][0], nef[mt][1], nef[mt][2], nef[mt][3], bt00, bt01);
                    mma_bf16(w2[hg][mt][1], nef[mt][0], nef[mt][1], nef[mt][2], nef[mt][3], bt10, bt11);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        float v = cs1[hg][nt][i];
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        v += __shfl_xor_sync(0xffffffffu, v, 8);
                        v += __shfl_xor_sync(0xffffffffu, v, 16);
                        c1r[hg][nt][i] += v;
                    }
            }
            put_w2(W2N);
        }
        {
            // partial A_q A_k^T over this warp's hidden units, straight from registers
            float s2[2][4] = {};
#pragma unroll
            for (int hg = 0; hg < 2; ++hg) {
                const uint32_t a0 = pack_bf16(aq[hg][0][0], aq[hg][0][1]), a1 = pack_bf16(aq[hg][0][2], aq[hg][0][3]);
                const uint32_t a2 = pack_bf16(aq[hg][1][0], aq[hg][1][1]), a3 = pack_bf16(aq[hg][1][2], aq[hg][1][3]);
                mma_bf16(s2[0], a0, a1, a2, a3, akp[hg][0], akp[hg][2]);  // key tokens 0-7
                mma_bf16(s2[1], a0, a1, a2, a3, akp[hg][1], akp[hg][3]);  // key tokens 8-15
            }
            float *sf = reinterpret_cast<float *>(gbase + C::S2F_OFF) + w * 16 * C::S2R;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                *reinterpret_cast<float2 *>(sf + g * C::S2R + 8 * nt + 2 * t4) = make_float2(s2[nt][0], s2[nt][1]);
                *reinterpret_cast<float2 *>(sf + (g + 8) * C::S2R + 8 * nt + 2 * t4) = make_float2(s2[nt][2], s2[nt][3]);
            }
        }
        __syncthreads();  // B3: A_q, partials visible; the stage's tiles are no longer read
        prev_t0 = J.t0;
        prev_c = J.c;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            c2r[nt][0] += cs2[nt][0];
            c2r[nt][1] += cs2[nt][1];
        }
        w2cur ^= 1;
    }

    if (prev_c > 0 && !*abort_flag) {  // the last chunk's outputs
        reduce_s2(prev_c);
        __syncthreads();
        if (w >= 4) {
            float pz[2][2][4] = {};
            col_product16(base + C::W2B_OFF + (uint32_t)((w2cur ^ 1) * M * C::W2R), AQ, pz);
            store_z(pz, base + C::NEB_OFF + (uint32_t)(((jb - 1) & 1) * 16 * C::ER), prev_t0, prev_c,
                    reinterpret_cast<const float *>(gbase + C::C2S_OFF) + ((jb - 1) & 1) * D);
        }
    }

    // ------------------------------------------------------------ final state
#pragma unroll
    for (int hg = 0; hg < 2; ++hg) {
        const int h0 = 32 * w + 16 * hg;
        if (p.W1o) {
            float *o = p.W1o + (size_t)bh * D * M;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int r = 8 * j + 2 * t4;
                o[(size_t)r * M + h0 + g] = w1[hg][j][0];
                o[(size_t)(r + 1) * M + h0 + g] = w1[hg][j][1];
                o[(size_t)r * M + h0 + g + 8] = w1[hg][j][2];
                o[(size_t)(r + 1) * M + h0 + g + 8] = w1[hg][j][3];
            }
        }
        if (p.c1o && g == 0) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 2; ++i) p.c1o[(size_t)bh * M + h0 + 8 * nt + 2 * t4 + i] = c1r[hg][nt][i];
        }
        if (p.W2o) {
            float *o = p.W2o + (size_t)bh * M * D;
#pragma unroll
            for (int mt = 0; mt < NK; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int hr = h0 + 8 * nt + 2 * t4, dc = 16 * mt + g;
                    o[(size_t)hr * D + dc] = w2[hg][mt][nt][0];
                    o[(size_t)(hr + 1) * D + dc] = w2[hg][mt][nt][1];
                    o[(size_t)hr * D + dc + 8] = w2[hg][mt][nt][2];
                    o[(size_t)(hr + 1) * D + dc + 8] = w2[hg][mt][nt][3];
                }
        }
    }
    if (p.c2o && g == 0 && w < 4) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            p.c2o[(size_t)bh * D + cc + 8 * nt + 2 * t4] = c2r[nt][0];
            p.c2o[(size_t)bh * D + cc + 8 * nt + 2 * t4 + 1] = c2r[nt][1];
        }
    }
    // make sure no copy is still landing in shared memory when the CTA ends
    if (warp == 0)
        for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
            if (!mbar_wait(bar_full + 8 * (j % NS), (j / NS) & 1, p.status, kSiteDrain)) break;
}

