// Compile-time Clebsch-Gordan tables and path enumeration for the channelwise tensor product.
//
// Everything here is constexpr C++20: the CUDA kernels are specialised per irreps
// configuration and read the CG records as compile-time constants (they become FFMA
// immediates), while the host side uses the same functions to export the tables through
// e3gb_table_info.
//
// CG construction: "e3j: An efficient and open-source backend for Euclidean equivariant
// operations on GPU and TPU", App. G.2, Eq. (22)-(25):
//   1. the top-spin vector |L L> = sum_m V_m |l1 m, l2 (L-m)> solves the eigen-equation
//      J^2 V = L(L+1) V (Eq. 25), a three-term recurrence in m solved from the lowest m;
//   2. |L M-1> is proportional to J_- |L M> with J_- = J_- (x) 1 + 1 (x) J_- (Leibniz rule);
//   3. normalised states give <l1 m1 l2 m2 | L M> in the complex (spin) basis.
// The real basis is that of the component-normalised real harmonics with m = -l..l
// (sin-type for m < 0, cos-type for m > 0, sqrt(3)(y,z,x) for l = 1):
//   Y_m^R = ((-1)^m Y^m + Y^-m)/sqrt2 (m > 0),  Y_-k^R = i (Y^-k - (-1)^k Y^k)/sqrt2 (k > 0).
// The real block is the change of basis of the complex one, made real by a global phase,
// scaled so that sum_{m1,m2} C[m1,m2,m3]^2 = 1 for every m3, with the sign fixed so that
// the first entry in row-major (m1, m2, m3) order is positive.
//
// Paths: every (x block, l2 <= sh_lmax, |l1-l2| <= l3 <= min(l1+l2, out_lmax)) triangle,
// ordered by (x block, l2, l3); output parity p1 (-1)^l2 (App. B.1 selection rule). Summed
// mode: one output block per distinct (l3, p3), ordered by l3, natural parity (-1)^l3 first;
// per-path mode: one output block per path.
#pragma once

#include <array>
#include <cstdint>

namespace e3gb {

constexpr int kLmax = 3;
constexpr int kMaxBlocks = 8;

constexpr double csqrt(double x) {
    if (x <= 0.0) return 0.0;
    double g = x > 1.0 ? x : 1.0;
    for (int i = 0; i < 200; ++i) {
        double n = 0.5 * (g + x / g);
        if (n == g) break;
        g = n;
    }
    return g;
}
constexpr double cabs(double x) { return x < 0 ? -x : x; }

// ladder coefficients c_{+-}(l, m) = sqrt(l(l+1) - m(m +- 1))
constexpr double cplus(int l, int m) { return csqrt(double(l * (l + 1) - m * (m + 1))); }
constexpr double cminus(int l, int m) { return csqrt(double(l * (l + 1) - m * (m - 1))); }

struct Block7 {
    double v[7][7][7] = {};   // [m1 + l1][m2 + l2][m3 + l3]
};

// <l1 m1 l2 m2 | L M> in the spin basis, by the ladder construction of App. G.2.
constexpr Block7 spin_cg(int l1, int l2, int L) {
    Block7 out{};
    if (L < (l1 > l2 ? l1 - l2 : l2 - l1) || L > l1 + l2) return out;
    // 1. top state: V_m for m1 = m, m2 = L - m
    double V[7] = {};
    const int mlo = (-l1 > L - l2) ? -l1 : L - l2;
    const int mhi = (l1 < L + l2) ? l1 : L + l2;
    V[mlo + l1] = 1.0;
    for (int m = mlo; m < mhi; ++m) {
        const int mp = L - m;
        const double diag = double(l1 * (l1 + 1) + l2 * (l2 + 1) + 2 * m * mp) - double(L * (L + 1));
        double rhs = diag * V[m + l1];
        if (m - 1 >= mlo) rhs += cplus(l1, m - 1) * cminus(l2, mp + 1) * V[m - 1 + l1];
        const double coef = cminus(l1, m + 1) * cplus(l2, mp - 1);
        V[m + 1 + l1] = -rhs / coef;
    }
    double n2 = 0;
    for (int m = mlo; m <= mhi; ++m) n2 += V[m + l1] * V[m + l1];
    const double inv = 1.0 / csqrt(n2);
    for (int m = mlo; m <= mhi; ++m) out.v[m + l1][L - m + l2][2 * L] = V[m + l1] * inv;
    // 2. lower: |L M-1> = J_- |L M> / c_-(L, M)
    for (int M = L; M > -L; --M) {
        const double nrm = 1.0 / cminus(L, M);
        for (int m1 = -l1; m1 <= l1; ++m1)
            for (int m2 = -l2; m2 <= l2; ++m2) {
                if (m1 + m2 != M - 1) continue;
                double s = 0;
                if (m1 + 1 <= l1) s += cminus(l1, m1 + 1) * out.v[m1 + 1 + l1][m2 + l2][M + L];
                if (m2 + 1 <= l2) s += cminus(l2, m2 + 1) * out.v[m1 + l1][m2 + 1 + l2][M + L];
                out.v[m1 + l1][m2 + l2][M - 1 + L] = s * nrm;
            }
    }
    return out;
}

struct Cx {
    double re = 0, im = 0;
};
constexpr Cx cmul(Cx a, Cx b) { return {a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re}; }
constexpr Cx conj(Cx a) { return {a.re, -a.im}; }

// U[m][mu]: real basis state m as a combination of spin states mu (two entries per row).
constexpr Cx Uent(int m, int mu) {
    const double r = 1.0 / csqrt(2.0);
    if (m == 0) return mu == 0 ? Cx{1, 0} : Cx{0, 0};
    if (m > 0) {
        if (mu == m) return Cx{(m % 2 ? -r : r), 0};
        if (mu == -m) return Cx{r, 0};
        return Cx{0, 0};
    }
    const int k = -m;
    if (mu == -k) return Cx{0, r};
    if (mu == k) return Cx{0, (k % 2 ? r : -r)};
    return Cx{0, 0};
}

// Real-basis block C[m1][m2][m3] (normalised, sign-fixed, zeros below 1e-12).
constexpr Block7 real_cg(int l1, int l2, int l3) {
    Block7 out{};
    const Block7 s = spin_cg(l1, l2, l3);
    Block7 re{}, im{};
    double nre = 0, nim = 0;
    for (int m1 = -l1; m1 <= l1; ++m1)
        for (int m2 = -l2; m2 <= l2; ++m2)
            for (int m3 = -l3; m3 <= l3; ++m3) {
                Cx acc{};
                for (int u1 = -l1; u1 <= l1; ++u1) {
                    const Cx a = conj(Uent(m1, u1));
                    if (a.re == 0 && a.im == 0) continue;
                    for (int u2 = -l2; u2 <= l2; ++u2) {
                        const Cx b = conj(Uent(m2, u2));
                        if (b.re == 0 && b.im == 0) continue;
                        const int u3 = u1 + u2;
                        if (u3 < -l3 || u3 > l3) continue;
                        const Cx c = Uent(m3, u3);
                        if (c.re == 0 && c.im == 0) continue;
                        const double g = s.v[u1 + l1][u2 + l2][u3 + l3];
                        const Cx t = cmul(cmul(a, b), c);
                        acc.re += t.re * g;
                        acc.im += t.im * g;
                    }
                }
                re.v[m1 + l1][m2 + l2][m3 + l3] = acc.re;
                im.v[m1 + l1][m2 + l2][m3 + l3] = acc.im;
                nre += acc.re * acc.re;
                nim += acc.im * acc.im;
            }
    const Block7& src = nre >= nim ? re : im;
    const double n = nre >= nim ? nre : nim;
    if (n == 0) return out;
    const double scale = csqrt(double(2 * l3 + 1) / n);
    double sign = 0;
    for (int m1 = 0; m1 < 2 * l1 + 1; ++m1)
        for (int m2 = 0; m2 < 2 * l2 + 1; ++m2)
            for (int m3 = 0; m3 < 2 * l3 + 1; ++m3) {
                double v = src.v[m1][m2][m3] * scale;
                if (cabs(v) < 1e-12) v = 0;
                if (sign == 0 && v != 0) sign = v > 0 ? 1 : -1;
                out.v[m1][m2][m3] = v;
            }
    for (int m1 = 0; m1 < 7; ++m1)
        for (int m2 = 0; m2 < 7; ++m2)
            for (int m3 = 0; m3 < 7; ++m3) out.v[m1][m2][m3] *= sign;
    return out;
}

// ------------------------------------------------------------------------------------------
// irreps configurations
// ------------------------------------------------------------------------------------------

// x irreps code: block i uses 4 bits at 4i: bit0-1 = l, bit2 = odd parity, bit3 = present.
constexpr uint32_t xblock(int l, int parity) { return uint32_t(8 | (parity < 0 ? 4 : 0) | l); }
constexpr int xcode_nblocks(uint32_t c) {
    int n = 0;
    while (n < kMaxBlocks && ((c >> (4 * n)) & 8u)) ++n;
    return n;
}
constexpr int xcode_l(uint32_t c, int i) { return int((c >> (4 * i)) & 3u); }
constexpr int xcode_p(uint32_t c, int i) { return ((c >> (4 * i)) & 4u) ? -1 : 1; }

struct PathInfo {
    int xblock, l1, p1, l2, l3, p3;
    int xoff, yoff, out_block, zoff;
};

struct OutBlock {
    int l, p;
};

constexpr int count_paths(uint32_t xc, int L2, int L3) {
    int n = 0;
    for (int i = 0; i < xcode_nblocks(xc); ++i) {
        const int l1 = xcode_l(xc, i);
        for (int l2 = 0; l2 <= L2; ++l2)
            for (int l3 = (l1 > l2 ? l1 - l2 : l2 - l1); l3 <= l1 + l2 && l3 <= L3; ++l3) ++n;
    }
    return n;
}

constexpr int out_order_key(int l, int p) { return 2 * l + (p == ((l & 1) ? -1 : 1) ? 0 : 1); }

template <int NP>
struct PathTable {
    std::array<PathInfo, NP> paths{};
    std::array<OutBlock, NP> outs{};
    int n_out = 0, d1 = 0, d2 = 0, D = 0;
};

template <int NP>
constexpr PathTable<NP> make_paths(uint32_t xc, int L2, int L3, bool per_path) {
    PathTable<NP> t{};
    int xoffs[kMaxBlocks] = {};
    int off = 0;
    for (int i = 0; i < xcode_nblocks(xc); ++i) {
        xoffs[i] = off;
        off += 2 * xcode_l(xc, i) + 1;
    }
    t.d1 = off;
    t.d2 = (L2 + 1) * (L2 + 1);
    int n = 0;
    for (int i = 0; i < xcode_nblocks(xc); ++i) {
        const int l1 = xcode_l(xc, i), p1 = xcode_p(xc, i);
        for (int l2 = 0; l2 <= L2; ++l2)
            for (int l3 = (l1 > l2 ? l1 - l2 : l2 - l1); l3 <= l1 + l2 && l3 <= L3; ++l3) {
                PathInfo p{};
                p.xblock = i; p.l1 = l1; p.p1 = p1; p.l2 = l2; p.l3 = l3;
                p.p3 = p1 * ((l2 & 1) ? -1 : 1);
                p.xoff = xoffs[i]; p.yoff = l2 * l2;
                t.paths[n++] = p;
            }
    }
    if (per_path) {
        for (int k = 0; k < NP; ++k) {
            t.outs[k] = OutBlock{t.paths[k].l3, t.paths[k].p3};
            t.paths[k].out_block = k;
        }
        t.n_out = NP;
    } else {
        // distinct (l3, p3) sorted by out_order_key
        int m = 0;
        for (int key = 0; key < 2 * (kLmax + 1); ++key)
            for (int k = 0; k < NP; ++k) {
                if (out_order_key(t.paths[k].l3, t.paths[k].p3) != key) continue;
                bool seen = false;
                for (int j = 0; j < m; ++j)
                    if (t.outs[j].l == t.paths[k].l3 && t.outs[j].p == t.paths[k].p3) seen = true;
                if (!seen) t.outs[m++] = OutBlock{t.paths[k].l3, t.paths[k].p3};
            }
        t.n_out = m;
        for (int k = 0; k < NP; ++k)
            for (int j = 0; j < m; ++j)
                if (t.outs[j].l == t.paths[k].l3 && t.outs[j].p == t.paths[k].p3) t.paths[k].out_block = j;
    }
    int zo[NP] = {};
    int z = 0;
    for (int j = 0; j < t.n_out; ++j) {
        zo[j] = z;
        z += 2 * t.outs[j].l + 1;
    }
    t.D = z;
    for (int k = 0; k < NP; ++k) t.paths[k].zoff = zo[t.paths[k].out_block];
    return t;
}

// One nonzero CG record of a path: C_p[m1][m2][m3] = c (m's are 0-based: m + l).
struct Rec {
    int path, m1, m2, m3;
    float c;
    double cd;
};

// A-entry: A_p[m3][m1] = sum_t c_t y[yoff + m2_t]; the y-contracted coupling of one edge.
struct AEnt {
    int path, m3, m1, nt;
    int m2[4];
    float c[4];
};

template <int NP>
constexpr int count_recs(const PathTable<NP>& t) {
    int n = 0;
    for (int k = 0; k < NP; ++k) {
        const Block7 b = real_cg(t.paths[k].l1, t.paths[k].l2, t.paths[k].l3);
        for (int a = 0; a < 2 * t.paths[k].l1 + 1; ++a)
            for (int c = 0; c < 2 * t.paths[k].l2 + 1; ++c)
                for (int d = 0; d < 2 * t.paths[k].l3 + 1; ++d)
                    if (b.v[a][c][d] != 0) ++n;
    }
    return n;
}

template <int NP>
constexpr int count_aents(const PathTable<NP>& t) {
    int n = 0;
    for (int k = 0; k < NP; ++k) {
        const Block7 b = real_cg(t.paths[k].l1, t.paths[k].l2, t.paths[k].l3);
        for (int d = 0; d < 2 * t.paths[k].l3 + 1; ++d)
            for (int a = 0; a < 2 * t.paths[k].l1 + 1; ++a) {
                bool any = false;
                for (int c = 0; c < 2 * t.paths[k].l2 + 1; ++c)
                    if (b.v[a][c][d] != 0) any = true;
                if (any) ++n;
            }
    }
    return n;
}

template <int NP, int NR>
constexpr std::array<Rec, NR> make_recs(const PathTable<NP>& t) {
    std::array<Rec, NR> r{};
    int n = 0;
    for (int k = 0; k < NP; ++k) {
        const Block7 b = real_cg(t.paths[k].l1, t.paths[k].l2, t.paths[k].l3);
        for (int a = 0; a < 2 * t.paths[k].l1 + 1; ++a)
            for (int c = 0; c < 2 * t.paths[k].l2 + 1; ++c)
                for (int d = 0; d < 2 * t.paths[k].l3 + 1; ++d)
                    if (b.v[a][c][d] != 0) r[n++] = Rec{k, a, c, d, float(b.v[a][c][d]), b.v[a][c][d]};
    }
    return r;
}

// A-entries ordered by path, then m3, then m1.
template <int NP, int NA>
constexpr std::array<AEnt, NA> make_aents(const PathTable<NP>& t) {
    std::array<AEnt, NA> r{};
    int n = 0;
    for (int k = 0; k < NP; ++k) {
        const Block7 b = real_cg(t.paths[k].l1, t.paths[k].l2, t.paths[k].l3);
        for (int d = 0; d < 2 * t.paths[k].l3 + 1; ++d)
            for (int a = 0; a < 2 * t.paths[k].l1 + 1; ++a) {
                AEnt e{};
                e.path = k; e.m3 = d; e.m1 = a; e.nt = 0;
                for (int c = 0; c < 2 * t.paths[k].l2 + 1; ++c)
                    if (b.v[a][c][d] != 0) {
                        if (e.nt < 4) {
                            e.m2[e.nt] = c;
                            e.c[e.nt] = float(b.v[a][c][d]);
                        }
                        ++e.nt;
                    }
                if (e.nt > 0) r[n++] = e;
            }
    }
    return r;
}

template <int NP, int NA>
constexpr int max_terms(const std::array<AEnt, NA>& a) {
    int m = 0;
    for (int i = 0; i < NA; ++i) m = a[i].nt > m ? a[i].nt : m;
    return m;
}

// Full compile-time description of one irreps configuration.
template <uint32_t XC, int L2_, int L3_, bool PP>
struct Config {
    static constexpr uint32_t xcode = XC;
    static constexpr int L2 = L2_, L3 = L3_;
    static constexpr bool per_path = PP;
    static constexpr int NP = count_paths(XC, L2_, L3_);
    static constexpr PathTable<NP> table = make_paths<NP>(XC, L2_, L3_, PP);
    static constexpr int D1 = table.d1, D2 = table.d2, D = table.D, NOUT = table.n_out;
    static constexpr int NR = count_recs(table);
    static constexpr int NA = count_aents(table);
    static constexpr std::array<Rec, NR> recs = make_recs<NP, NR>(table);
    static constexpr std::array<AEnt, NA> aents = make_aents<NP, NA>(table);
    static_assert(max_terms<NP, NA>(aents) <= 4, "more than 4 m2 terms in one A entry");
    static_assert(NP > 0, "configuration with no paths");
};

}  // namespace e3gb
