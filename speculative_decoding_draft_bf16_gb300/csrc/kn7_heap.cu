// kn7_heap.cu -- best-first heap with parent-conditioned edge scores, and the
// TDES edge-score table.
//
// [DARTree] tree-construction ablation (Table 2): the exact sequential
// alternative to DARTree corrects the children of each popped node and updates
// a heap.  [GRAFT] "Inference": a max-heap orders prefixes by the sum of their
// TDES edge scores and the best prefix joins the tree until the budget is met;
// "Target-distilled edge scoring": the edge scorer f(p, c, d) =
// w . ReLU(W [g_p(e_p); g_c(e_c); e_d] + b) + b0 with a learned scale s.
//
// Edge score of child j (position d) under a parent whose token is candidate i
// of position d-1 (the root at d = 1): t = lp_d[j] + E[d-1][i][j], minus the
// DARTree log-normaliser z[d-1][i] when given, in fp32; a path score adds t to
// its parent's score.  Because every parent is a candidate of the previous
// position, the children's order under a parent (t desc, j asc) depends only
// on (d, i): it is one row of an order table, computed once per row.  The heap
// is DDTree's best-first search with those orders in place of the ranks: pop
// the best prefix (score desc, then its descriptor of order positions, a prefix
// first), push its first child and its next sibling.  Nodes are written in pop
// order (parents before children).
//
// One CTA per request.  All warps first compute every order row when they all
// fit in shared memory (the usual sizes), else only the root's; warp 0 then
// runs the B pops alone, computing a missing row when a node needing it is
// popped.  The frontier (at most B + 1 entries, each carrying its parent's
// order row and score) lives in shared memory, cut into blocks of 32 slots
// whose maxima the lanes keep in registers, so a pop is a warp max and one
// ballot; ties on the score go to the smaller descriptor, found by walking
// both parent chains.  The popped slot takes one of the pushes.  A per-request
// budget (budget[b], clamped to [1, B]) bounds the pops of that request.
//
// TDES table (kn8): the projections depend only on the token, so the inputs
// are the per-token first-layer rows Ap = W_p g_p(e), Ac = W_c g_c(e) and the
// per-depth rows Dd = W_d e_d + b; per edge a = (Ap[p] + Ac[c]) + Dd[d-1],
// r = max(a, 0), f = sum_h w_h r_h (serial fma from 0) + b0, E = s * f.
#include "dt_device.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT7 = 256;
constexpr int NW7 = NT7 / 32;
constexpr int NT8 = 256;

DT_DI uint32_t ordf(float t) {
    const uint32_t u = __float_as_uint(t);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
DT_DI float unordf(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k); }

struct Kn7Smem {
    float* lp;        // [L*K] candidate log-probabilities
    int* id;          // [L*K] candidate tokens
    int* rowmap;      // [L*K] order row of (child position d, parent rank i) at (d-1)*K + i, -1 none
    uint16_t* ord;    // [cap_rows][K] children in edge order (candidate ranks)
    float* ts;        // [cap_rows][K] their edge scores
    unsigned long long* keys;  // [NW7][K] sort scratch, one slice per warp
    float* fs;        // [B+1] frontier: path score
    int4* fe;         // [B+1] frontier: parent node, (depth << 16) | order position, parent's order
                      //       row, parent's score (bits)
    int* npar;        // [Mmax] emitted nodes
    int* nord;
    int* ndep;
    int* nrank;
    int* ntok;
    float* nsc;
    int* misc;        // [0]: rows in use
};

__host__ __device__ inline int kn7_total_rows(int L, int K) { return 1 + (L - 1) * K; }
__host__ __device__ inline int kn7_cap_rows(int L, int K, int B) {
    const int t = kn7_total_rows(L, K);
    return t < B + 1 ? t : B + 1;
}

__host__ __device__ inline size_t kn7_layout(int L, int K, int B, int Mmax, Kn7Smem* S, unsigned char* base) {
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + 15) & ~(size_t)15;
        return at;
    };
    const int cap = kn7_cap_rows(L, K, B);
    const size_t o_lp = take((size_t)L * K * 4), o_id = take((size_t)L * K * 4), o_rm = take((size_t)L * K * 4);
    const size_t o_ord = take((size_t)cap * K * 2), o_ts = take((size_t)cap * K * 4);
    const size_t o_keys = take((size_t)NW7 * K * 8);
    const size_t o_fs = take((size_t)(B + 1) * 4), o_fe = take((size_t)(B + 1) * 16);
    const size_t o_np = take((size_t)Mmax * 4), o_no = take((size_t)Mmax * 4), o_nd = take((size_t)Mmax * 4);
    const size_t o_nk = take((size_t)Mmax * 4), o_nt = take((size_t)Mmax * 4);
    const size_t o_ns = take((size_t)Mmax * 4), o_misc = take(16);
    if (S) {
        S->lp = (float*)(base + o_lp);
        S->id = (int*)(base + o_id);
        S->rowmap = (int*)(base + o_rm);
        S->ord = (uint16_t*)(base + o_ord);
        S->ts = (float*)(base + o_ts);
        S->keys = (unsigned long long*)(base + o_keys);
        S->fs = (float*)(base + o_fs);
        S->fe = (int4*)(base + o_fe);
        S->npar = (int*)(base + o_np);
        S->nord = (int*)(base + o_no);
        S->ndep = (int*)(base + o_nd);
        S->nrank = (int*)(base + o_nk);
        S->ntok = (int*)(base + o_nt);
        S->nsc = (float*)(base + o_ns);
        S->misc = (int*)(base + o_misc);
    }
    return o;
}

// Order row `r` for the children at position d (1-based) of parent rank i,
// computed by one warp: edge scores, then each child's place by counting the
// children ahead of it (score desc, rank asc).
DT_DI void make_row(const Kn7Smem& S, int r, int d, int i, int K, const float* tab, bool term, const float* z,
                    unsigned long long* keys) {
    const int lane = threadIdx.x & 31;
    for (int j = lane; j < K; j += 32) {
        float t = S.lp[(d - 1) * K + j];
        if (tab) t = __fadd_rn(t, term ? tab[((size_t)(d - 1) * K + i) * K + j] : 0.f);
        if (z) t = __fsub_rn(t, z[(size_t)(d - 1) * K + i]);
        keys[j] = ((unsigned long long)ordf(t) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)j);
    }
    __syncwarp();
    for (int j = lane; j < K; j += 32) {
        const unsigned long long kj = keys[j];
        int pos = 0;
        for (int q = 0; q < K; ++q) pos += keys[q] > kj;
        S.ord[(size_t)r * K + pos] = (uint16_t)j;
        S.ts[(size_t)r * K + pos] = unordf((uint32_t)(kj >> 32));
    }
    __syncwarp();
}

// Descriptor order of frontier entries (parent pa, position ja) and (pb, jb):
// lexicographic on the order positions from the root, a prefix first.
DT_DI bool desc_less(const Kn7Smem& S, int pa, int ja, int pb, int jb) {
    const int la = S.ndep[pa] + 1, lb = S.ndep[pb] + 1;
    int da = la, db = lb;
    int xa = ja, ua = pa, xb = jb, ub = pb;
    while (da > db) { xa = S.nord[ua]; ua = S.npar[ua]; --da; }
    while (db > da) { xb = S.nord[ub]; ub = S.npar[ub]; --db; }
    int res = 0;  // decided at the level nearest the root where they differ
    for (;;) {
        if (xa != xb) res = xa < xb ? -1 : 1;
        if (ua == ub) break;
        xa = S.nord[ua]; ua = S.npar[ua];
        xb = S.nord[ub]; ub = S.npar[ub];
    }
    if (res) return res < 0;
    return la < lb;
}

// Frontier entry a before entry b?
DT_DI bool entry_before(const Kn7Smem& S, int a, float sa, int b, float sb) {
    if (sa != sb) return sa > sb;
    return desc_less(S, S.fe[a].x, S.fe[a].y & 0xFFFF, S.fe[b].x, S.fe[b].y & 0xFFFF);
}

__global__ void __launch_bounds__(NT7, 1) kn7_kernel(int L, int V, int K, int B, const int32_t* __restrict__ budget,
                                                  int Mmax,
                                                  const float* __restrict__ cand_lp,
                                                  const int32_t* __restrict__ cand_id,
                                                  const float* __restrict__ table,
                                                  const int32_t* __restrict__ root_tok,
                                                  const float* __restrict__ znorm, int32_t* __restrict__ o_tok,
                                                  int32_t* __restrict__ o_par, int32_t* __restrict__ o_dep,
                                                  int32_t* __restrict__ o_rank, float* __restrict__ o_score,
                                                  int32_t* __restrict__ o_n, int32_t* __restrict__ status) {
    extern __shared__ __align__(128) unsigned char smem[];
    Kn7Smem S;
    kn7_layout(L, K, B, Mmax, &S, smem);
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    dt_pdl_trigger();
    dt_pdl_wait();  // candidate tables, edge table and normalisers come from earlier kernels
    const size_t cb = (size_t)b * L * K;
    for (int x = tid; x < L * K; x += NT7) {
        S.lp[x] = cand_lp[cb + x];
        S.id[x] = cand_id[cb + x];
        S.rowmap[x] = -1;
    }
    const float* tab = table ? table + cb * K : nullptr;
    const float* z = znorm ? znorm + cb : nullptr;
    const int rt = root_tok ? root_tok[b] : -1;
    const bool root_term = rt >= 0 && rt < V;
    const int total = kn7_total_rows(L, K), cap = kn7_cap_rows(L, K, B);
    __syncthreads();
    // order rows: all of them when they fit, else the root's now and the rest on demand
    const int pre = total <= cap ? total : 1;
    for (int r = wid; r < pre; r += NW7) {
        const int d = r == 0 ? 1 : 2 + (r - 1) / K, i = r == 0 ? 0 : (r - 1) % K;
        make_row(S, r, d, i, K, tab, d > 1 || root_term, z, S.keys + (size_t)wid * K);
        if (lane == 0) S.rowmap[(d - 1) * K + i] = r;
    }
    __syncthreads();

    if (wid == 0) {
        int nrows = pre;
        // the root and its first child
        if (lane == 0) {
            S.npar[0] = -1; S.nord[0] = 0; S.ndep[0] = 0; S.nrank[0] = -1; S.ntok[0] = -1;
            S.nsc[0] = 0.f;
            S.fs[0] = __fadd_rn(0.f, S.ts[0]);
            S.fe[0] = make_int4(0, 1 << 16, 0, __float_as_int(0.f));  // first child of the root, order row 0
        }
        __syncwarp();
        // Block maxima: the frontier is cut into blocks of 32 slots; lane l keeps
        // the largest score key of blocks l and l + 32 (0: empty).  A pop is a
        // warp max over them and one ballot inside the winning block; only the
        // blocks a pop changes are refreshed.  Equal best scores (rare outside
        // coarse logits) go to the full comparison with descriptors.
        uint32_t bk0 = 0, bk1 = 0;
        auto skey = [&](int x) { return ordf(__fadd_rn(S.fs[x], 0.f)); };  // -0 and +0 alike
        auto refresh = [&](int blk, int nfr) {
            const int x = blk * 32 + lane;
            const uint32_t m = __reduce_max_sync(0xffffffffu, x < nfr ? skey(x) : 0u);
            if (lane == (blk & 31)) {
                if (blk < 32) bk0 = m;
                else bk1 = m;
            }
        };
        int nf = 1, n = 0;
        refresh(0, nf);
        const int Bq = budget ? min(B, max(1, budget[b])) : B;  // this request's budget
        const bool all_rows = pre == total;  // row of (position d + 1, parent rank c): 1 + (d - 1) * K + c
        while (n < Bq && nf > 0) {
            if (n + 1 >= Mmax) break;  // the host checks max_nodes > B; never taken
            const uint32_t g = __reduce_max_sync(0xffffffffu, bk0 > bk1 ? bk0 : bk1);
            const unsigned h0 = __ballot_sync(0xffffffffu, bk0 == g), h1 = __ballot_sync(0xffffffffu, bk1 == g);
            int best = -1;
            if (__popc(h0) + __popc(h1) == 1) {
                const int blk = h0 ? __ffs(h0) - 1 : 32 + __ffs(h1) - 1;
                const int xl = blk * 32 + lane;
                const unsigned hit = __ballot_sync(0xffffffffu, xl < nf && skey(xl) == g);
                if (__popc(hit) == 1) best = blk * 32 + __ffs(hit) - 1;
            }
            if (best < 0) {  // several entries share the best score: descriptor order decides
                float bs = 0.f;
                for (int x = lane; x < nf; x += 32) {
                    const float sx = S.fs[x];
                    if (best < 0 || entry_before(S, x, sx, best, bs)) { best = x; bs = sx; }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const int ob = __shfl_xor_sync(0xffffffffu, best, o);
                    const float os = __shfl_xor_sync(0xffffffffu, bs, o);
                    if (ob >= 0 && (best < 0 || entry_before(S, ob, os, best, bs))) { best = ob; bs = os; }
                }
            }
            const int x = best;
            const float bs = S.fs[x];
            const int4 ent = S.fe[x];
            const int p = ent.x, j = ent.y & 0xFFFF, d = ent.y >> 16, rowp = ent.z;
            const int c = S.ord[rowp * K + j];
            const int m = ++n;
            int r = -1;  // order row of m's children
            if (d < L) {
                if (all_rows) {
                    r = 1 + (d - 1) * K + c;
                } else {
                    r = S.rowmap[d * K + c];
                    if (r < 0) {
                        r = nrows++;
                        make_row(S, r, d + 1, c, K, tab, true, z, S.keys);
                        if (lane == 0) S.rowmap[d * K + c] = r;
                    }
                }
            }
            const bool sib = j + 1 < K, kid = r >= 0;
            __syncwarp();
            // the popped slot takes the sibling, else the first child; the other is appended
            const int last = nf - 1;
            const int kid_slot = sib ? nf : x;
            if (lane == 0) {
                S.npar[m] = p; S.nord[m] = j; S.ndep[m] = d; S.nrank[m] = c; S.ntok[m] = S.id[(d - 1) * K + c];
                S.nsc[m] = bs;
                if (sib) {
                    S.fs[x] = __fadd_rn(__int_as_float(ent.w), S.ts[rowp * K + j + 1]);
                    S.fe[x] = make_int4(p, ent.y + 1, rowp, ent.w);
                }
                if (kid) {
                    S.fs[kid_slot] = __fadd_rn(bs, S.ts[r * K]);
                    S.fe[kid_slot] = make_int4(m, (d + 1) << 16, r, __float_as_int(bs));
                }
                if (!sib && !kid && x != last) {  // nothing to push: the last entry fills the slot
                    S.fs[x] = S.fs[last];
                    S.fe[x] = S.fe[last];
                }
            }
            nf = (sib && kid) ? nf + 1 : ((sib || kid) ? nf : last);
            __syncwarp();
            // blocks touched: the popped slot's, and the appended or vacated slot's
            const int bx = x >> 5;
            const int bo = (sib && kid) ? (nf - 1) >> 5 : ((!sib && !kid) ? last >> 5 : bx);
            refresh(bx, nf);
            if (bo != bx) refresh(bo, nf);
        }
        if (lane == 0) S.misc[0] = n;
    }
    __syncthreads();
    const int nn = S.misc[0] + 1;
    const size_t ob = (size_t)b * Mmax;
    for (int v = tid; v < nn; v += NT7) {
        o_tok[ob + v] = S.ntok[v];
        o_par[ob + v] = S.npar[v];
        o_dep[ob + v] = S.ndep[v];
        o_rank[ob + v] = S.nrank[v];
        o_score[ob + v] = S.nsc[v];
    }
    if (tid == 0) {
        o_n[b] = nn;
        int bits = 0;
        for (int x = 0; x < L; ++x)
            if (S.lp[x * K] != S.lp[x * K]) bits |= DT_DEV_TIMEOUT;  // stage 1 flagged this row
        if (z)
            for (int x = 0; x < L * K; ++x)
                if (z[x] != z[x]) bits |= DT_DEV_TIMEOUT;  // the normaliser kernel flagged this row
        status[b] = bits;
    }
}

// TDES edge table: block (position d, request b); thread per edge (i, j).
__global__ void __launch_bounds__(NT8) kn8_kernel(int L, int K, int H, int V, const float* __restrict__ Ap,
                                                  const float* __restrict__ Ac, const float* __restrict__ Dd,
                                                  const float* __restrict__ w, float b0, float s,
                                                  const int32_t* __restrict__ root_tok,
                                                  const int32_t* __restrict__ cand_id, float* __restrict__ table) {
    extern __shared__ __align__(16) float sm8[];
    const int d = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int Hp = H | 1;  // odd row stride: conflict-free reads of different rows
    float* Ps = sm8;
    float* Cs = Ps + (size_t)K * Hp;
    float* ds = Cs + (size_t)K * Hp;
    float* ws = ds + H;
    dt_pdl_trigger();
    dt_pdl_wait();
    int np;
    if (d == 0) {
        const int rt = root_tok ? root_tok[b] : -1;
        if (rt < 0 || rt >= V) return;  // no term at depth 1
        np = 1;
        for (int h = tid; h < H; h += NT8) Ps[h] = Ap[(size_t)rt * H + h];
    } else {
        np = K;
        for (int t = tid; t < K * H; t += NT8) {
            const int i = t / H, h = t % H;
            Ps[i * Hp + h] = Ap[(size_t)cand_id[((size_t)b * L + d - 1) * K + i] * H + h];
        }
    }
    for (int t = tid; t < K * H; t += NT8) {
        const int j = t / H, h = t % H;
        Cs[j * Hp + h] = Ac[(size_t)cand_id[((size_t)b * L + d) * K + j] * H + h];
    }
    for (int h = tid; h < H; h += NT8) {
        ds[h] = Dd[(size_t)d * H + h];
        ws[h] = w[h];
    }
    __syncthreads();
    float* out = table + ((size_t)b * L + d) * K * K;
    for (int t = tid; t < np * K; t += NT8) {
        const int i = t / K, j = t % K;
        const float* pr = Ps + (size_t)i * Hp;
        const float* cr = Cs + (size_t)j * Hp;
        float acc = 0.f;
        for (int h = 0; h < H; ++h) {
            const float a = __fadd_rn(__fadd_rn(pr[h], cr[h]), ds[h]);
            acc = __fmaf_rn(ws[h], a > 0.f ? a : 0.f, acc);
        }
        out[i * K + j] = __fmul_rn(s, __fadd_rn(acc, b0));
    }
}

}  // namespace

size_t dt_kn7_smem_bytes(int L, int K, int B, int Mmax) { return kn7_layout(L, K, B, Mmax, nullptr, nullptr); }

cudaError_t dt_kn7_launch(int batch, int L, int V, int K, int B, const int32_t* budget, int Mmax, const float* cand_lp,
                          const int32_t* cand_id, const float* table, const int32_t* root_tok, const float* znorm,
                          int32_t* tok, int32_t* parent, int32_t* depth, int32_t* rank, float* score,
                          int32_t* n_nodes, int32_t* status, cudaStream_t st) {
    const size_t sm = dt_kn7_smem_bytes(L, K, B, Mmax);
    if (sm > (size_t)227 * 1024 || K > 65535 || Mmax < B + 1) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kn7_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    DtLaunch lc(dim3(batch), dim3(NT7), sm, st);
    return cudaLaunchKernelEx(&lc.cfg, kn7_kernel, L, V, K, B, budget, Mmax, cand_lp, cand_id, table, root_tok, znorm, tok,
                              parent, depth, rank, score, n_nodes, status);
}

size_t dt_kn8_smem_bytes(int K, int H) { return ((size_t)2 * K * (H | 1) + 2 * (size_t)H) * 4; }

cudaError_t dt_kn8_launch(int batch, int L, int V, int K, int H, const float* Ap, const float* Ac, const float* Dd,
                          const float* w, float b0, float s, const int32_t* root_tok, const int32_t* cand_id,
                          float* table, cudaStream_t st) {
    const size_t sm = dt_kn8_smem_bytes(K, H);
    if (sm > (size_t)227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kn8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    DtLaunch lc(dim3(L, batch), dim3(NT8), sm, st);
    return cudaLaunchKernelEx(&lc.cfg, kn8_kernel, L, K, H, V, Ap, Ac, Dd, w, b0, s, root_tok, cand_id, table);
}
