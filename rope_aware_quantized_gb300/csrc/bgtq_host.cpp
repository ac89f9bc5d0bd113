// Host side of the Block-GTQ packed-cache library: allocation, plan (codec
// tables, Lloyd-Max codebooks, lane layout), and the C ABI entry points.
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — English
// abstract (energy score per RoPE block, greedy integer widths by marginal
// gain, uniform TQ-MSE values, packed-cache serving path) and the paper
// review §1 Key Terms / §3 Method & Key Results (TQ-MSE rotates then
// quantises; the greedy uses the 4^-b distortion rate).
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <algorithm>
#include <numeric>

#include "bgtq_internal.h"

namespace bgtq {

static thread_local std::string g_error;

int set_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_error = buf;
    return code;
}

// ----------------------------------------------------------------------------- half <-> double

static double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = std::ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = std::ldexp((double)(m | 1024), e - 25);
    return sign ? -v : v;
}

// Nearest-even fp16 of a double in the normal fp16 range (all centroids are).
static uint16_t double_to_half_bits(double x) {
    if (x == 0.0) return std::signbit(x) ? 0x8000 : 0;
    uint16_t sign = x < 0 ? 0x8000 : 0;
    double a = std::fabs(x);
    int e;
    std::frexp(a, &e);            // a = f * 2^e, f in [0.5, 1)
    double ulp = std::ldexp(1.0, e - 11);
    double q = std::nearbyint(a / ulp);  // exact scaling; ties to even
    double r = q * ulp;
    std::frexp(r, &e);
    int biased = e - 1 + 15;
    int mant = (int)(std::ldexp(r, 11 - e) - 1024.0);
    return (uint16_t)(sign | (biased << 10) | mant);
}

// ----------------------------------------------------------------------------- SplitMix64 signs

static uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static int rot_sign(uint64_t seed, int head, int tag, int j) {
    uint64_t key = seed ^ ((uint64_t)head << 16) ^ ((uint64_t)tag << 8) ^ (uint64_t)j;
    return (splitmix64(key) >> 63) ? -1 : 1;
}

// ----------------------------------------------------------------------------- RoPE blocks

static void block_dims(int rope_layout, int i, int* lo, int* hi) {
    if (rope_layout == 0) {
        *lo = i;
        *hi = i + kNB;
    } else {
        *lo = 2 * i;
        *hi = 2 * i + 1;
    }
}

// ----------------------------------------------------------------------------- Lloyd-Max codebook
// Lloyd-Max quantiser of N(0,1) with 2^b levels.  Newton's method on the
// thresholds of "threshold = midpoint of neighbouring centroids, centroid =
// conditional mean of its cell", from the high-rate point density.

static double npdf(double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI); }
static double ncdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }
static double nsf(double x) { return 0.5 * std::erfc(x / std::sqrt(2.0)); }

static double ncdf_inv(double p) {  // bisection; only used for the starting point
    double lo = -40.0, hi = 40.0;
    for (int i = 0; i < 200; ++i) {
        double mid = 0.5 * (lo + hi);
        if (ncdf(mid) < p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

static void cell_means(const std::vector<double>& t, std::vector<double>& c, std::vector<double>& mass) {
    int n = (int)t.size() + 1;
    c.assign(n, 0.0);
    mass.assign(n, 0.0);
    for (int k = 0; k < n; ++k) {
        double a = k == 0 ? -INFINITY : t[k - 1];
        double b = k == n - 1 ? INFINITY : t[k];
        double m = a > 0 ? nsf(a) - nsf(b) : ncdf(b) - ncdf(a);
        mass[k] = m;
        c[k] = (npdf(a) - npdf(b)) / m;
    }
}

static void lloyd_max(int bits, std::vector<double>& cent) {
    int n = 1 << bits;
    if (n == 2) {
        double c = std::sqrt(2.0 / M_PI);
        cent = {-c, c};
        return;
    }
    std::vector<double> t(n - 1), c, mass;
    for (int k = 1; k < n; ++k) t[k - 1] = std::sqrt(3.0) * ncdf_inv((double)k / n);
    std::vector<double> dl(n - 1), dd(n - 1), du(n - 1), rhs(n - 1);
    for (int it = 0; it < 200; ++it) {
        cell_means(t, c, mass);
        // Jacobian of F_k = t_k - (c_k + c_{k+1})/2
        for (int k = 0; k < n - 1; ++k) {
            // cell k = [t_{k-1}, t_k], cell k+1 = [t_k, t_{k+1}]
            double bk = t[k];
            double dck_db = npdf(bk) * (bk - c[k]) / mass[k];          // d c_k / d t_k
            double dck1_da = npdf(bk) * (c[k + 1] - bk) / mass[k + 1];  // d c_{k+1} / d t_k
            dd[k] = 1.0 - 0.5 * (dck_db + dck1_da);
            rhs[k] = -(t[k] - 0.5 * (c[k] + c[k + 1]));
            // dF_k / dt_{k-1} = -0.5 d c_k / d t_{k-1}
            if (k > 0) {
                double a = t[k - 1];
                dl[k] = -0.5 * npdf(a) * (c[k] - a) / mass[k];
            } else {
                dl[k] = 0.0;
            }
            // dF_k / dt_{k+1} = -0.5 d c_{k+1} / d t_{k+1}
            if (k < n - 2) {
                double b = t[k + 1];
                du[k] = -0.5 * npdf(b) * (b - c[k + 1]) / mass[k + 1];
            } else {
                du[k] = 0.0;
            }
        }
        // Thomas algorithm
        int m = n - 1;
        std::vector<double> cp(m), dp(m);
        cp[0] = du[0] / dd[0];
        dp[0] = rhs[0] / dd[0];
        for (int k = 1; k < m; ++k) {
            double den = dd[k] - dl[k] * cp[k - 1];
            cp[k] = du[k] / den;
            dp[k] = (rhs[k] - dl[k] * dp[k - 1]) / den;
        }
        std::vector<double> step(m);
        step[m - 1] = dp[m - 1];
        for (int k = m - 2; k >= 0; --k) step[k] = dp[k] - cp[k] * step[k + 1];
        double mx = 0.0;
        for (int k = 0; k < m; ++k) {
            t[k] += step[k];
            mx = std::max(mx, std::fabs(step[k]));
        }
        std::vector<double> ts(t);
        for (int k = 0; k < m; ++k) t[k] = 0.5 * (ts[k] - ts[m - 1 - k]);
        if (mx < 1e-13) break;
    }
    cell_means(t, c, mass);
    cent.resize(n);
    for (int k = 0; k < n; ++k) cent[k] = 0.5 * (c[k] - c[n - 1 - k]);
}

// ----------------------------------------------------------------------------- allocation

static int alloc_impl(const uint16_t* calib, int64_t n, int bits_per_key, int b_max, int rope_layout,
                      uint8_t* bits_out, double* energy_out) {
    double s[kNB];
    for (int i = 0; i < kNB; ++i) {
        int lo, hi;
        block_dims(rope_layout, i, &lo, &hi);
        double acc = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            double a = half_to_double(calib[t * kD + lo]);
            double b = half_to_double(calib[t * kD + hi]);
            acc = (acc + a * a) + b * b;
        }
        s[i] = acc / (double)n;
    }
    int b[kNB] = {0};
    for (int step = 0; step < bits_per_key / 2; ++step) {
        int best = -1;
        double best_gain = 0.0;
        for (int i = 0; i < kNB; ++i) {
            if (b[i] >= b_max) continue;
            double g = std::ldexp(s[i], -2 * b[i]);
            if (best < 0 || g > best_gain) {
                best = i;
                best_gain = g;
            }
        }
        b[best] += 1;
    }
    for (int i = 0; i < kNB; ++i) {
        bits_out[i] = (uint8_t)b[i];
        if (energy_out) energy_out[i] = s[i];
    }
    return BGTQ_OK;
}

// ----------------------------------------------------------------------------- lane layout of the K record
// Pairs (codec coords 2m, 2m+1) are ranked by (width desc, index asc); lanes
// 0..2 take the first 16-subset, in the order ((rank - lane) mod 4, rank),
// whose widths sum to 16*bK; lane 3 takes the rest.  Slots inside a lane
// alternate between the even and odd ranks of the lane's width order.

static bool lane_layout(const int wd[kNB], int bk, uint8_t slot_pair[4][16], uint16_t slot_off[4][16]) {
    const int target = 16 * bk;
    int rank_of[kNB];
    std::vector<int> ord(kNB);
    std::iota(ord.begin(), ord.end(), 0);
    std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) {
        if (wd[a] != wd[b]) return wd[a] > wd[b];
        return a < b;
    });
    for (int r = 0; r < kNB; ++r) rank_of[ord[r]] = r;
    std::vector<bool> used(kNB, false);
    std::vector<int> lanes[4];
    for (int t = 0; t < 3; ++t) {
        std::vector<int> order;
        for (int m = 0; m < kNB; ++m)
            if (!used[m]) order.push_back(m);
        std::sort(order.begin(), order.end(), [&](int a, int b) {
            int ka = ((rank_of[a] - t) % 4 + 4) % 4, kb = ((rank_of[b] - t) % 4 + 4) % 4;
            if (ka != kb) return ka < kb;
            return rank_of[a] < rank_of[b];
        });
        int n = (int)order.size();
        // feas[i][k][s]: k items summing to s can be picked from order[i..]
        std::vector<uint8_t> feas((size_t)(n + 1) * 17 * (target + 1), 0);
        auto F = [&](int i, int k, int s) -> uint8_t& { return feas[((size_t)i * 17 + k) * (target + 1) + s]; };
        F(n, 0, 0) = 1;
        for (int i = n - 1; i >= 0; --i) {
            int w = wd[order[i]];
            for (int k = 0; k <= 16; ++k)
                for (int s = 0; s <= target; ++s) {
                    uint8_t v = F(i + 1, k, s);
                    if (!v && k > 0 && s >= w) v = F(i + 1, k - 1, s - w);
                    F(i, k, s) = v;
                }
        }
        if (!F(0, 16, target)) return false;
        int k = 16, s = target;
        for (int i = 0; i < n && k > 0; ++i) {
            int m = order[i], w = wd[m];
            if (s >= w && F(i + 1, k - 1, s - w)) {
                lanes[t].push_back(m);
                used[m] = true;
                --k;
                s -= w;
            }
        }
    }
    for (int m = 0; m < kNB; ++m)
        if (!used[m]) lanes[3].push_back(m);
    for (int t = 0; t < 4; ++t) {
        std::vector<int> a = lanes[t];
        if ((int)a.size() != 16) return false;
        std::stable_sort(a.begin(), a.end(), [&](int x, int y) {
            if (wd[x] != wd[y]) return wd[x] > wd[y];
            return x < y;
        });
        int o = 0;
        for (int s = 0; s < 16; ++s) {
            int m = s < 8 ? a[2 * s] : a[2 * (s - 8) + 1];
            slot_pair[t][s] = (uint8_t)m;
            slot_off[t][s] = (uint16_t)o;
            o += 2 * wd[m];
        }
        if (o != 32 * bk) return false;
    }
    return true;
}

// ----------------------------------------------------------------------------- plan

static void free_dev(bgtq_plan* p) {
    if (p->dev.heads) cudaFree(p->dev.heads);
    if (p->dev.cent) cudaFree(p->dev.cent);
    if (p->dev.thr) cudaFree(p->dev.thr);
    if (p->dev.img_src) cudaFree(p->dev.img_src);
    if (p->dev.cells) cudaFree(p->dev.cells);
    p->dev = DevTables{};
}

static int build_head(bgtq_plan* p, int h, const uint8_t* bits, const double* s) {
    HeadTab& ht = p->heads[h];
    std::memset(&ht, 0, sizeof(ht));
    // codec order: width classes (desc), blocks ascending, cut into pieces
    struct Piece { int size, w; std::vector<int> coords; };
    std::vector<Piece> pieces;
    for (int w = kWMax; w >= 1; --w) {
        std::vector<int> coords;
        for (int i = 0; i < kNB; ++i)
            if (bits[i] == w) {
                int lo, hi;
                block_dims(p->rope_layout, i, &lo, &hi);
                coords.push_back(lo);
                coords.push_back(hi);
            }
        size_t pos = 0;
        for (int e = 7; e >= 1; --e) {
            size_t size = (size_t)1 << e;
            if (coords.size() & size) {
                pieces.push_back({(int)size, w, std::vector<int>(coords.begin() + pos, coords.begin() + pos + size)});
                pos += size;
            }
        }
    }
    std::stable_sort(pieces.begin(), pieces.end(), [](const Piece& a, const Piece& b) {
        if (a.size != b.size) return a.size > b.size;
        return a.w > b.w;
    });
    int dim_block[kD];
    for (int i = 0; i < kNB; ++i) {
        int lo, hi;
        block_dims(p->rope_layout, i, &lo, &hi);
        dim_block[lo] = i;
        dim_block[hi] = i;
    }
    int j = 0;
    p->piece[h].assign(kD, 0);
    p->sign_k8[h].assign(kD, 0);
    p->sign_v8[h].assign(kD, 0);
    for (const Piece& pc : pieces) {
        int lg = 0;
        while ((1 << lg) < pc.size) ++lg;
        for (int c : pc.coords) {
            ht.perm[j] = (uint8_t)c;
            ht.width[j] = (uint8_t)pc.w;
            ht.plog2[j] = (uint8_t)lg;
            p->piece[h][j] = (uint8_t)pc.size;
            double si = s[dim_block[c]];
            ht.whiten[j] = si == 0.0 ? 1.0f : (float)std::sqrt(2.0 / si);
            ht.dewhiten[j] = (float)std::sqrt(si / 2.0);
            ht.inv_sqrt[j] = (float)(1.0 / std::sqrt((double)pc.size));
            int sg = rot_sign(p->seed, h, 0, j);
            ht.sign_k[j] = (float)sg;
            p->sign_k8[h][j] = (int8_t)sg;
            ++j;
        }
    }
    ht.n_coded = j;
    for (int v = 0; v < kD; ++v) {
        int sg = rot_sign(p->seed, h, 1, v);
        ht.sign_v[v] = (float)sg;
        p->sign_v8[h][v] = (int8_t)sg;
    }
    // lane layout of the K record
    int wd[kNB];
    for (int m = 0; m < kNB; ++m) wd[m] = 2 * m < ht.n_coded ? ht.width[2 * m] : 0;
    uint16_t off[4][16];
    if (!lane_layout(wd, p->bk, ht.slot_pair, off))
        return set_error(BGTQ_ERR_UNSUPPORTED, "head %d: no balanced lane layout for this allocation", h);
    p->slot_off[h].assign(64, 0);
    ht.max_w = 0;
    for (int m = 0; m < kNB; ++m) ht.max_w = std::max(ht.max_w, wd[m]);
    // decode lookup recipes (KSlot): slots 0..7 read the lane slice shifted
    // left by 7 bits (a field at slice bit o sits at window bit o + 7); slots
    // 8..15 read the words (1, 2) for bK = 3, else (0, 1) or the single word.
    // The slots of a lane are sorted by width, the even ranks first, so the
    // first eight fields end by bit 16 bK + 8 and the last eight start at bit
    // 16 bK or later: every field fits its window at a shift >= 0.  The table
    // base of the single tables is set per plan (upload_plan), as it depends
    // on the widest code of all heads.
    ht.n_wide = 0;
    for (int t = 0; t < 4; ++t) {
        int lead = 0;
        for (int r = 0; r < 16; ++r) {
            const int sl = (r & 1) ? 8 + r / 2 : r / 2;  // width order 0, 8, 1, 9, ...
            if (wd[ht.slot_pair[t][sl]] > kPairTableMaxW) lead = r + 1;
        }
        ht.n_wide = std::max(ht.n_wide, lead);
    }
    for (int t = 0; t < 4; ++t)
        for (int sl = 0; sl < 16; ++sl) {
            const int m = ht.slot_pair[t][sl];
            const int w = wd[m];
            const int o = off[t][sl];
            p->slot_off[h][t * 16 + sl] = (uint16_t)o;
            ht.pair_bit[m] = (uint16_t)(32 * p->bk * t + o);
            KSlot& k = ht.kslot[t][sl];
            if (p->bk > 3) continue;  // no decode instance reads records of more than 3 words per lane
            const int sh = sl < 8 ? o : (p->bk == 3 ? o - 39 : o - 7);
            const int end = sl < 8 ? o + 7 + 2 * w : (p->bk == 3 ? o - 32 : o) + 2 * w;
            if (sh < 0 || end > 64 || (p->bk == 1 && sl >= 8 && end > 32))
                return set_error(BGTQ_ERR_UNSUPPORTED, "head %d: K slot (%d, %d) outside its decode window", h, t, sl);
            if (w <= kPairTableMaxW) {
                k.sh = (uint32_t)sh;
                k.mask = ((1u << (2 * w)) - 1u) << 7;
                k.base = (1u << (2 * w)) << 7;
                k.wsh = 0;
            } else if (w <= kLaneTableMaxW) {
                k.sh = (uint32_t)sh;
                k.mask = ((1u << w) - 1u) << 7;
                k.base = (uint32_t)single_base(w) << 7;
                k.wsh = (uint32_t)w;
            } else {  // shared table, 4-byte stride: the code at bit 2
                k.sh = (uint32_t)sh + 5;
                k.mask = ((1u << w) - 1u) << 2;
                k.base = kSharedTable;  // | byte offset, set per plan (the region follows the per-lane tables)
                k.wsh = (uint32_t)w;
            }
        }
    return BGTQ_OK;
}

// Decode table source for codes up to width ws: lane_entries(ws) words (the
// kernel stores 32 copies of each, one per lane), then shared_words(ws) words.
static void build_image_source(bgtq_plan* p, int ws) {
    p->img_ws = ws;
    p->img_src.assign(kImageMaxWords, 0);
    auto hb = [&](int w, int c) -> uint32_t {
        const float x = p->cent[w][c];
        return x == 0.0f ? 0u : (uint32_t)double_to_half_bits(x);
    };
    for (int w = 0; w <= kPairTableMaxW; ++w) {
        const int n = 1 << (2 * w), mask = (1 << w) - 1;
        for (int f = 0; f < n; ++f) p->img_src[(1 << (2 * w)) + f] = hb(w, f & mask) | (hb(w, f >> w) << 16);
    }
    for (int w = kPairTableMaxW + 1; w <= std::min(ws, kLaneTableMaxW); ++w)
        for (int c = 0; c < (1 << w); ++c) p->img_src[single_base(w) + c] = hb(w, c) | (hb(w, c) << 16);
    const int le = lane_entries(ws);
    for (int w = kLaneTableMaxW + 1; w <= ws; ++w)
        for (int c = 0; c < (1 << w); ++c) p->img_src[le + shared_word(w, ws) + c] = hb(w, c) | (hb(w, c) << 16);
}

static int build_codebooks(bgtq_plan* p) {
    for (int w = 0; w <= kWMax; ++w) {
        p->cent[w].clear();
        p->thr[w].clear();
        if (w == 0) {
            p->cent[0] = {0.0f};
            continue;
        }
        std::vector<double> c;
        lloyd_max(w, c);
        std::vector<double> ch(c.size());
        for (size_t k = 0; k < c.size(); ++k) ch[k] = half_to_double(double_to_half_bits(c[k]));
        for (size_t k = 0; k < c.size(); ++k) p->cent[w].push_back((float)ch[k]);
        for (size_t k = 0; k + 1 < c.size(); ++k) p->thr[w].push_back((float)(0.5 * (ch[k] + ch[k + 1])));
    }
    return BGTQ_OK;
}

// Code-search cell tables.  The code of a quotient u at width w is the number
// of width-w thresholds <= u.  The bulk encoder maps u to a cell by
// cell(u) = round(s * sat(a u + b)) (two correctly rounded fused
// multiply-adds, the second adding 1.5 * 2^23 so that the integer is the low
// bits of the result), a non-decreasing function of u.  A threshold whose cell
// is below cell(u) is then <= u and one whose cell is above is > u; so when
// no two thresholds share a cell, the code is base(c) + [t_c <= u] for
// c = cell(u), with base(c) the number of thresholds in the cells below c and
// t_c the threshold in c (+inf if none).  The cell count is raised until every
// threshold has a cell of its own, checked with the arithmetic of the device.
static uint32_t f2u(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

static float u2f(uint32_t u) {
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

static int cell_of(float u, float a, float b, float s) {
    float v = std::fmaf(u, a, b);
    v = v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);  // sat (no NaN reaches here)
    return (int)(f2u(std::fmaf(v, s, 12582912.0f)) - kCellMagicBits);
}

static int build_cells(bgtq_plan* p) {
    std::vector<uint32_t> hdr(kCellHdr, 0u), ent;
    for (int w = 0; w <= kWMax; ++w) {
        const std::vector<float>& t = p->thr[w];
        const int n = (int)t.size();
        float a = 0.0f, b = 0.0f, s = 0.0f;
        std::vector<int> cell(n);
        if (n > 0) {
            double gap = 1.0;
            for (int i = 0; i + 1 < n; ++i) gap = std::min(gap, (double)t[i + 1] - (double)t[i]);
            if (!(gap > 0.0)) return set_error(BGTQ_ERR_UNSUPPORTED, "width %d: repeated threshold", w);
            const double lo = (double)t[0] - gap, hi = (double)t[n - 1] + gap;
            bool ok = false;
            for (int cells = (int)std::ceil((hi - lo) / (0.9 * gap)) + 1; cells <= kCellMaxEntries; cells += cells / 16 + 1) {
                a = (float)(1.0 / (hi - lo));
                b = (float)(-lo / (hi - lo));
                s = (float)(cells - 1);
                ok = true;
                for (int i = 0; i < n && ok; ++i) {
                    cell[i] = cell_of(t[i], a, b, s);
                    ok = cell[i] >= 0 && cell[i] < cells && (i == 0 || cell[i] > cell[i - 1]);
                }
                if (ok) break;
            }
            if (!ok) return set_error(BGTQ_ERR_UNSUPPORTED, "width %d: no cell table", w);
        }
        const int cells = (int)s + 1;
        hdr[4 * w] = f2u(a);
        hdr[4 * w + 1] = f2u(b);
        hdr[4 * w + 2] = f2u(s);
        hdr[4 * w + 3] = (uint32_t)(ent.size() / 2);
        for (int c = 0, i = 0; c < cells; ++c) {
            while (i < n && cell[i] < c) ++i;  // i = thresholds in cells below c
            ent.push_back(i < n && cell[i] == c ? f2u(t[i]) : f2u(INFINITY));
            ent.push_back((uint32_t)i);
        }
    }
    if (ent.size() / 2 > (size_t)kCellMaxEntries) return set_error(BGTQ_ERR_UNSUPPORTED, "cell tables too large");
    p->cells = hdr;
    p->cells.insert(p->cells.end(), ent.begin(), ent.end());
    return BGTQ_OK;
}

// The code of u at width w through the cell tables (host copy of the bulk
// encoder's search; the tests compare it with a plain threshold count).
static int cell_code(const bgtq_plan* p, int w, float u) {
    const uint32_t* h = p->cells.data() + 4 * w;
    const int c = cell_of(u, u2f(h[0]), u2f(h[1]), u2f(h[2]));
    const uint32_t* e = p->cells.data() + kCellHdr + 2 * ((size_t)h[3] + (size_t)c);
    return (int)e[1] + (u2f(e[0]) <= u ? 1 : 0);
}

template <class T>
static cudaError_t upload(T** dst, const T* src, size_t n) {
    cudaError_t e = cudaMalloc((void**)dst, n * sizeof(T));
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice);
}

static int upload_plan(bgtq_plan* p) {
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "device attribute: %s", cudaGetErrorString(e));
    std::vector<float> cent(9 * 256, 0.0f), thr(9 * 256, 0.0f);
    for (int w = 0; w <= kWMax; ++w) {
        std::copy(p->cent[w].begin(), p->cent[w].end(), cent.begin() + 256 * w);
        std::copy(p->thr[w].begin(), p->thr[w].end(), thr.begin() + 256 * w);
    }
    if ((e = upload(&p->dev.heads, p->heads.data(), p->heads.size())) != cudaSuccess ||
        (e = upload(&p->dev.cent, cent.data(), cent.size())) != cudaSuccess ||
        (e = upload(&p->dev.thr, thr.data(), thr.size())) != cudaSuccess ||
        (e = upload(&p->dev.img_src, p->img_src.data(), p->img_src.size())) != cudaSuccess ||
        (e = upload(&p->dev.cells, p->cells.data(), p->cells.size())) != cudaSuccess) {
        free_dev(p);
        return set_error(BGTQ_ERR_CUDA, "plan upload: %s", cudaGetErrorString(e));
    }
    return BGTQ_OK;
}

static int check_plan(const bgtq_plan* p) {
    if (!p) return set_error(BGTQ_ERR_INVALID_ARG, "plan is NULL");
    if (p->flags & BGTQ_PLAN_HOST_ONLY) return set_error(BGTQ_ERR_INVALID_ARG, "plan was built host-only");
    return BGTQ_OK;
}

int check_cache(const bgtq_plan* p, const bgtq_cache* c) {
    if (!c || !c->k_codes || !c->k_norm || !c->v_codes || !c->v_norm)
        return set_error(BGTQ_ERR_INVALID_ARG, "cache descriptor or one of its buffers is NULL");
    if (c->capacity <= 0 || (c->capacity & 1)) return set_error(BGTQ_ERR_INVALID_ARG, "capacity must be even and > 0");
    if ((reinterpret_cast<uintptr_t>(c->k_codes) & 15) || (reinterpret_cast<uintptr_t>(c->v_codes) & 15))
        return set_error(BGTQ_ERR_INVALID_ARG, "k_codes and v_codes must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(c->k_norm) & 3) || (reinterpret_cast<uintptr_t>(c->v_norm) & 3))
        return set_error(BGTQ_ERR_INVALID_ARG, "k_norm and v_norm must be 4-byte aligned");
    if (c->recent < 0 || c->recent > c->capacity)
        return set_error(BGTQ_ERR_INVALID_ARG, "recent must be in [0, capacity]");
    if (c->recent > 0 && (!c->k_recent || (reinterpret_cast<uintptr_t>(c->k_recent) & 15)))
        return set_error(BGTQ_ERR_INVALID_ARG, "k_recent must be a 16-byte aligned buffer when recent > 0");
    if (c->page_table) {
        const int64_t P = c->page_tokens;
        if (P < 16 || P > (1 << 20) || (P & (P - 1)))
            return set_error(BGTQ_ERR_INVALID_ARG, "page_tokens must be a power of two in [16, 2^20]");
        if (c->max_pages < 1 || c->n_pages < 1 || c->n_pages > INT32_MAX)
            return set_error(BGTQ_ERR_INVALID_ARG, "max_pages and n_pages must be >= 1 (n_pages < 2^31)");
        if (c->capacity != c->max_pages * P)
            return set_error(BGTQ_ERR_INVALID_ARG, "a paged cache needs capacity == max_pages * page_tokens");
        if (reinterpret_cast<uintptr_t>(c->page_table) & 3)
            return set_error(BGTQ_ERR_INVALID_ARG, "page_table must be 4-byte aligned");
        if (c->capacity > (int64_t)1 << 21)
            return set_error(BGTQ_ERR_INVALID_ARG, "a paged cache holds at most 2^21 positions per sequence");
    }
    if (c->capacity > INT32_MAX) return set_error(BGTQ_ERR_INVALID_ARG, "capacity must be < 2^31");
    (void)p;
    return BGTQ_OK;
}

}  // namespace bgtq

using namespace bgtq;

extern "C" {

const char* bgtq_last_error(void) { return g_error.c_str(); }

int bgtq_alloc_bits(const uint16_t* calib, int64_t n, int head_dim, int bits_per_key, int b_max, int rope_layout,
                    uint8_t* bits_out, double* energy_out) {
    if (!calib || !bits_out) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (head_dim != kD) return set_error(BGTQ_ERR_UNSUPPORTED, "head_dim must be 128");
    if (n <= 0) return set_error(BGTQ_ERR_INVALID_ARG, "need n > 0 calibration keys");
    if (b_max < 1 || b_max > kWMax) return set_error(BGTQ_ERR_INVALID_ARG, "b_max must be in 1..8");
    if (bits_per_key < 0 || (bits_per_key & 1)) return set_error(BGTQ_ERR_INVALID_ARG, "bits_per_key must be even and >= 0");
    if (bits_per_key / 2 > kNB * b_max) return set_error(BGTQ_ERR_INVALID_ARG, "budget exceeds 64 * b_max");
    if (rope_layout != 0 && rope_layout != 1) return set_error(BGTQ_ERR_INVALID_ARG, "rope_layout must be 0 or 1");
    return alloc_impl(calib, n, bits_per_key, b_max, rope_layout, bits_out, energy_out);
}

int bgtq_plan_create(bgtq_plan** out, int head_dim, int n_kv_heads, int group, int bits_per_key, int v_bits,
                     const uint8_t* block_bits, const double* energy, uint64_t seed, int rope_layout, int flags) {
    if (!out || !block_bits || !energy) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    *out = nullptr;
    if (head_dim != kD) return set_error(BGTQ_ERR_UNSUPPORTED, "head_dim must be 128");
    if (n_kv_heads < 1 || n_kv_heads > 4096) return set_error(BGTQ_ERR_INVALID_ARG, "n_kv_heads out of range");
    if (group < 1 || group > 8) return set_error(BGTQ_ERR_UNSUPPORTED, "group (query heads per KV head) must be 1..8");
    if (bits_per_key <= 0 || bits_per_key % 128 || bits_per_key > 128 * kWMax)
        return set_error(BGTQ_ERR_INVALID_ARG, "bits_per_key must be a multiple of 128 in [128, 1024]");
    if (v_bits < 1 || v_bits > kPairMaxW) return set_error(BGTQ_ERR_UNSUPPORTED, "v_bits must be 1..5");
    if (rope_layout != 0 && rope_layout != 1) return set_error(BGTQ_ERR_INVALID_ARG, "rope_layout must be 0 or 1");
    for (int h = 0; h < n_kv_heads; ++h) {
        int sum = 0;
        for (int i = 0; i < kNB; ++i) {
            int b = block_bits[h * kNB + i];
            if (b > kWMax) return set_error(BGTQ_ERR_INVALID_ARG, "head %d block %d: width > 8", h, i);
            sum += b;
        }
        if (2 * sum != bits_per_key)
            return set_error(BGTQ_ERR_INVALID_ARG, "head %d: widths use %d bits, budget is %d", h, 2 * sum, bits_per_key);
    }
    bgtq_plan* p = new bgtq_plan();
    p->H = n_kv_heads;
    p->G = group;
    p->bits_per_key = bits_per_key;
    p->bk = bits_per_key / 128;
    p->bv = v_bits;
    p->rope_layout = rope_layout;
    p->seed = seed;
    p->flags = flags;
    p->in_bits.assign(block_bits, block_bits + (size_t)n_kv_heads * kNB);
    p->in_energy.assign(energy, energy + (size_t)n_kv_heads * kNB);
    p->heads.resize(n_kv_heads);
    p->sign_k8.resize(n_kv_heads);
    p->sign_v8.resize(n_kv_heads);
    p->piece.resize(n_kv_heads);
    p->slot_off.resize(n_kv_heads);
    int rc = build_codebooks(p);
    if (rc == BGTQ_OK) rc = build_cells(p);
    for (int h = 0; rc == BGTQ_OK && h < n_kv_heads; ++h) rc = build_head(p, h, block_bits + h * kNB, energy + h * kNB);
    if (rc == BGTQ_OK) {
        // decode tables: widest code of all heads (keys) and of the values
        int ws = p->bv > kPairTableMaxW ? p->bv : 0;
        for (const HeadTab& ht : p->heads) ws = std::max(ws, ht.max_w);
        build_image_source(p, ws);
        for (HeadTab& ht : p->heads)
            for (int t = 0; t < 4; ++t)
                for (int sl = 0; sl < 16; ++sl) {
                    KSlot& k = ht.kslot[t][sl];
                    if (k.base & kSharedTable)
                        k.base = kSharedTable | (uint32_t)(lane_entries(ws) * 128 + 4 * shared_word((int)k.wsh, ws));
                }
    }
    if (rc == BGTQ_OK && !(flags & BGTQ_PLAN_HOST_ONLY)) rc = upload_plan(p);
    if (rc != BGTQ_OK) {
        delete p;
        return rc;
    }
    *out = p;
    return BGTQ_OK;
}

// ---- plan serialization: the defining inputs, versioned and checksummed
// (every table is a deterministic function of them).  Little-endian:
//   "BGTQPLAN" | u32 version | u32 H, G, bits_per_key, v_bits, rope_layout |
//   u64 seed | u8 widths[H][64] | f64 energies[H][64] | u64 FNV-1a of all
//   preceding bytes

}  // extern "C"

namespace {

constexpr char kPlanMagic[8] = {'B', 'G', 'T', 'Q', 'P', 'L', 'A', 'N'};
constexpr uint32_t kPlanVersion = 1;
constexpr size_t kPlanHeader = 8 + 4 + 5 * 4 + 8;

uint64_t fnv1a(const uint8_t* d, size_t n) {
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= d[i];
        h *= 1099511628211ull;
    }
    return h;
}

void put_le(uint8_t*& o, uint64_t v, int nbytes) {
    for (int i = 0; i < nbytes; ++i) *o++ = (uint8_t)(v >> (8 * i));
}

uint64_t get_le(const uint8_t*& i, int nbytes) {
    uint64_t v = 0;
    for (int k = 0; k < nbytes; ++k) v |= (uint64_t)(*i++) << (8 * k);
    return v;
}

}  // namespace

extern "C" {

int bgtq_plan_save(const bgtq_plan* p, void* buf, size_t capacity, size_t* bytes) {
    if (!p || !bytes) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    const size_t n = kPlanHeader + (size_t)p->H * kNB * (1 + 8) + 8;
    *bytes = n;
    if (!buf) return BGTQ_OK;
    if (capacity < n) return set_error(BGTQ_ERR_INVALID_ARG, "buffer holds %zu bytes, the plan needs %zu", capacity, n);
    uint8_t* o = static_cast<uint8_t*>(buf);
    std::memcpy(o, kPlanMagic, 8);
    o += 8;
    put_le(o, kPlanVersion, 4);
    put_le(o, (uint32_t)p->H, 4);
    put_le(o, (uint32_t)p->G, 4);
    put_le(o, (uint32_t)p->bits_per_key, 4);
    put_le(o, (uint32_t)p->bv, 4);
    put_le(o, (uint32_t)p->rope_layout, 4);
    put_le(o, p->seed, 8);
    for (uint8_t b : p->in_bits) *o++ = b;
    for (double e : p->in_energy) {
        uint64_t u;
        std::memcpy(&u, &e, 8);
        put_le(o, u, 8);
    }
    const uint64_t h = fnv1a(static_cast<const uint8_t*>(buf), (size_t)(o - static_cast<uint8_t*>(buf)));
    put_le(o, h, 8);
    return BGTQ_OK;
}

int bgtq_plan_load(bgtq_plan** out, const void* buf, size_t bytes, int flags) {
    if (!out || !buf) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    *out = nullptr;
    const uint8_t* b = static_cast<const uint8_t*>(buf);
    if (bytes < kPlanHeader + 8 || std::memcmp(b, kPlanMagic, 8) != 0)
        return set_error(BGTQ_ERR_INVALID_ARG, "not a serialized Block-GTQ plan");
    const uint8_t* i = b + 8;
    const uint32_t version = (uint32_t)get_le(i, 4);
    if (version != kPlanVersion)
        return set_error(BGTQ_ERR_UNSUPPORTED, "plan format version %u (this library reads version %u)", version,
                         kPlanVersion);
    const int H = (int)get_le(i, 4), G = (int)get_le(i, 4), bpk = (int)get_le(i, 4), bv = (int)get_le(i, 4);
    const int layout = (int)get_le(i, 4);
    const uint64_t seed = get_le(i, 8);
    if (H < 1 || H > 4096) return set_error(BGTQ_ERR_INVALID_ARG, "serialized plan: head count %d out of range", H);
    const size_t n = kPlanHeader + (size_t)H * kNB * (1 + 8) + 8;
    if (bytes < n) return set_error(BGTQ_ERR_INVALID_ARG, "serialized plan truncated (%zu of %zu bytes)", bytes, n);
    const uint8_t* ce = b + n - 8;
    if (get_le(ce, 8) != fnv1a(b, n - 8)) return set_error(BGTQ_ERR_INVALID_ARG, "serialized plan: checksum mismatch");
    std::vector<uint8_t> bits(i, i + (size_t)H * kNB);
    i += (size_t)H * kNB;
    std::vector<double> energy((size_t)H * kNB);
    for (double& e : energy) {
        const uint64_t u = get_le(i, 8);
        std::memcpy(&e, &u, 8);
    }
    return bgtq_plan_create(out, kD, H, G, bpk, bv, bits.data(), energy.data(), seed, layout, flags);
}

int bgtq_plan_destroy(bgtq_plan* p) {
    if (!p) return BGTQ_OK;
    free_dev(p);
    delete p;
    return BGTQ_OK;
}

int bgtq_plan_get_head(const bgtq_plan* p, int head, bgtq_head_tables* out) {
    if (!p || !out) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (head < 0 || head >= p->H) return set_error(BGTQ_ERR_INVALID_ARG, "head out of range");
    const HeadTab& ht = p->heads[head];
    out->n_coded = ht.n_coded;
    out->perm = ht.perm;
    out->width = ht.width;
    out->piece = p->piece[head].data();
    out->sign_k = p->sign_k8[head].data();
    out->sign_v = p->sign_v8[head].data();
    out->whiten = ht.whiten;
    out->dewhiten = ht.dewhiten;
    out->slot_pair = &ht.slot_pair[0][0];
    out->slot_offset = p->slot_off[head].data();
    return BGTQ_OK;
}

int bgtq_plan_get_codebook(const bgtq_plan* p, int width, const float** cent, const float** thr, int* n_levels) {
    if (!p || !cent || !thr || !n_levels) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (width < 0 || width > kWMax) return set_error(BGTQ_ERR_INVALID_ARG, "width out of range");
    *cent = p->cent[width].data();
    *thr = p->thr[width].data();
    *n_levels = (int)p->cent[width].size();
    return BGTQ_OK;
}

int bgtq_plan_code(const bgtq_plan* p, int width, const float* u, int64_t n, int32_t* codes) {
    if (!p || (n > 0 && (!u || !codes))) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (width < 0 || width > kWMax || n < 0) return set_error(BGTQ_ERR_INVALID_ARG, "width or count out of range");
    for (int64_t i = 0; i < n; ++i) {
        if (std::isnan(u[i])) return set_error(BGTQ_ERR_INVALID_ARG, "NaN quotient at %lld", (long long)i);
        codes[i] = cell_code(p, width, u[i]);
    }
    return BGTQ_OK;
}

int bgtq_cache_bytes(const bgtq_plan* p, int batch, int64_t capacity, size_t* kb, size_t* vb, size_t* nb) {
    if (!p || !kb || !vb || !nb) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (batch < 0 || capacity < 0 || (capacity & 1)) return set_error(BGTQ_ERR_INVALID_ARG, "bad batch/capacity");
    size_t units = (size_t)batch * p->H;
    *kb = units * (size_t)capacity * 16 * p->bk;
    *vb = units * (size_t)(capacity / 2) * 32 * p->bv;
    *nb = units * (size_t)capacity * sizeof(float);
    return BGTQ_OK;
}

int bgtq_quantize_append(const bgtq_plan* p, void* stream, const void* k, const void* v, int batch, int t_new,
                         const int32_t* pos_start, const bgtq_cache* c, int32_t* status) {
    // the descriptor first: its checks read no device memory
    int rc = check_cache(p, c);
    if (rc) return rc;
    if ((rc = check_plan(p))) return rc;
    if (batch < 0 || t_new < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and t_new must be >= 0");
    if (batch == 0 || t_new == 0) return BGTQ_OK;
    if (!k || !v || !pos_start) return set_error(BGTQ_ERR_INVALID_ARG, "NULL input pointer");
    if (c->recent > 0 && ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 7))
        return set_error(BGTQ_ERR_INVALID_ARG, "k and v must be 8-byte aligned when the cache has a recent-key buffer");
    cudaError_t e = launch_quantize_append(*p, (cudaStream_t)stream, k, v, batch, t_new, pos_start, *c, status);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "quantize_append launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}

int bgtq_decode_attn_workspace(const bgtq_plan* p, int batch, int64_t max_len, size_t* bytes) {
    if (!p || !bytes) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (batch < 0 || max_len < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and max_len must be >= 0");
    *bytes = decode_workspace_bytes(*p, batch, decode_split(*p, batch, max_len));
    return BGTQ_OK;
}

int bgtq_decode_attn(const bgtq_plan* p, void* stream, const void* q, const bgtq_cache* c, const int32_t* seq_lens,
                     int64_t max_len, int batch, void* out, int out_dtype, float scale, void* ws, size_t ws_bytes,
                     int32_t* status) {
    int rc = check_plan(p);
    if (rc) return rc;
    if ((rc = check_cache(p, c))) return rc;
    if (batch < 0 || max_len < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and max_len must be >= 0");
    if (batch == 0) return BGTQ_OK;
    if (!q || !seq_lens || !out || !ws) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (out_dtype != 0 && out_dtype != 1) return set_error(BGTQ_ERR_INVALID_ARG, "out_dtype must be 0 (half) or 1 (float)");
    if (p->bk > 3) return set_error(BGTQ_ERR_UNSUPPORTED, "decode supports bits_per_key <= 384");
    if (p->bv > 4) return set_error(BGTQ_ERR_UNSUPPORTED, "decode supports v_bits <= 4");
    if (!(scale > 0.0f) || !std::isfinite(scale)) return set_error(BGTQ_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (max_len > c->capacity) max_len = c->capacity;
    SplitPlan sp = decode_split(*p, batch, max_len);
    size_t need = decode_workspace_bytes(*p, batch, sp);
    if (ws_bytes < need) return set_error(BGTQ_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    cudaError_t e = launch_decode(*p, (cudaStream_t)stream, q, *c, seq_lens, batch, sp, out, out_dtype, scale, ws, status);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "decode_attn launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}

int bgtq_decode_step(const bgtq_plan* p, void* stream, const void* q, const void* k_new, const void* v_new,
                     const int32_t* pos_new, const bgtq_cache* c, const int32_t* seq_lens, int64_t max_len, int batch,
                     void* out, int out_dtype, float scale, void* ws, size_t ws_bytes, int32_t* status) {
    int rc = check_plan(p);
    if (rc) return rc;
    if ((rc = check_cache(p, c))) return rc;
    if (batch < 0 || max_len < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and max_len must be >= 0");
    if (batch == 0) return BGTQ_OK;
    if (!q || !k_new || !v_new || !pos_new || !seq_lens || !out || !ws)
        return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 7)
        return set_error(BGTQ_ERR_INVALID_ARG, "k_new and v_new must be 8-byte aligned");
    if (out_dtype != 0 && out_dtype != 1) return set_error(BGTQ_ERR_INVALID_ARG, "out_dtype must be 0 (half) or 1 (float)");
    if (p->bk > 3) return set_error(BGTQ_ERR_UNSUPPORTED, "decode supports bits_per_key <= 384");
    if (p->bv > 4) return set_error(BGTQ_ERR_UNSUPPORTED, "decode supports v_bits <= 4");
    if (!(scale > 0.0f) || !std::isfinite(scale)) return set_error(BGTQ_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (max_len > c->capacity) max_len = c->capacity;
    SplitPlan sp = decode_split(*p, batch, max_len);
    size_t need = decode_workspace_bytes(*p, batch, sp);
    if (ws_bytes < need) return set_error(BGTQ_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    cudaError_t e = launch_decode(*p, (cudaStream_t)stream, q, *c, seq_lens, batch, sp, out, out_dtype, scale, ws, status,
                                  k_new, v_new, pos_new);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "decode_step launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}

int bgtq_prefill_attn(const bgtq_plan* p, void* stream, const void* q, const void* k, const void* v, int batch,
                      int t, const bgtq_cache* c, void* out, int out_dtype, float scale, int32_t* status) {
    // the descriptor and the arguments first (none of these checks reads
    // device memory), the plan's device tables last
    if (!p) return set_error(BGTQ_ERR_INVALID_ARG, "plan is NULL");
    int rc = check_cache(p, c);
    if (rc) return rc;
    if (batch < 0 || t < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and t must be >= 0");
    if (t > c->capacity) return set_error(BGTQ_ERR_CAPACITY, "t = %d exceeds the cache capacity", t);
    if (batch == 0 || t == 0) return BGTQ_OK;
    if (!q || !k || !v || !out) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
        return set_error(BGTQ_ERR_INVALID_ARG, "q, k and v must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(out) & 15) return set_error(BGTQ_ERR_INVALID_ARG, "out must be 16-byte aligned");
    if (out_dtype != 0 && out_dtype != 1) return set_error(BGTQ_ERR_INVALID_ARG, "out_dtype must be 0 (half) or 1 (float)");
    if (!(scale > 0.0f) || !std::isfinite(scale)) return set_error(BGTQ_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (batch > 65535) return set_error(BGTQ_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    if ((uint64_t)batch * p->H * p->G * (uint64_t)t + 128 >= (1ull << 31))
        return set_error(BGTQ_ERR_UNSUPPORTED, "batch * query heads * t must stay below 2^31 - 128");
    if ((rc = check_plan(p))) return rc;
    cudaError_t e = launch_prefill(*p, (cudaStream_t)stream, q, k, v, batch, t, *c, out, out_dtype, scale, status);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}

int bgtq_prefill_chunk_workspace(const bgtq_plan* p, int batch, int64_t max_prefix, size_t* bytes) {
    if (!p || !bytes) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (batch < 0 || max_prefix < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and max_prefix must be >= 0");
    *bytes = prefill_chunk_workspace_bytes(*p, batch, max_prefix);
    return BGTQ_OK;
}

int bgtq_prefill_chunk_attn(const bgtq_plan* p, void* stream, const void* q, const void* k, const void* v, int batch,
                            int t, const int32_t* pos_start, int64_t max_prefix, const bgtq_cache* c, void* out,
                            int out_dtype, float scale, void* ws, size_t ws_bytes, int32_t* status) {
    if (!p) return set_error(BGTQ_ERR_INVALID_ARG, "plan is NULL");
    int rc = check_cache(p, c);
    if (rc) return rc;
    if (batch < 0 || t < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and c must be >= 0");
    if (max_prefix < 0) return set_error(BGTQ_ERR_INVALID_ARG, "max_prefix must be >= 0");
    if (t > c->capacity) return set_error(BGTQ_ERR_CAPACITY, "c = %d exceeds the cache capacity", t);
    if (max_prefix > c->capacity) return set_error(BGTQ_ERR_CAPACITY, "max_prefix exceeds the cache capacity");
    if (batch == 0 || t == 0) return BGTQ_OK;
    if (!q || !k || !v || !out || !pos_start) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
        return set_error(BGTQ_ERR_INVALID_ARG, "q, k and v must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(out) & 15) return set_error(BGTQ_ERR_INVALID_ARG, "out must be 16-byte aligned");
    if (out_dtype != 0 && out_dtype != 1) return set_error(BGTQ_ERR_INVALID_ARG, "out_dtype must be 0 (half) or 1 (float)");
    if (!(scale > 0.0f) || !std::isfinite(scale)) return set_error(BGTQ_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (c->recent > 0)
        return set_error(BGTQ_ERR_UNSUPPORTED, "chunked prefill onto a cache with a recent-key buffer is not supported");
    if ((uint64_t)batch * p->H * p->G * (uint64_t)t + 128 >= (1ull << 31) ||
        (uint64_t)batch * p->H * (uint64_t)(max_prefix + 128) + 128 >= (1ull << 31))
        return set_error(BGTQ_ERR_UNSUPPORTED, "batch * query heads * c and batch * heads * max_prefix must stay below 2^31");
    const size_t need = prefill_chunk_workspace_bytes(*p, batch, max_prefix);
    if (ws_bytes < need) return set_error(BGTQ_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    if (need > 0 && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)))
        return set_error(BGTQ_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device buffer");
    if ((rc = check_plan(p))) return rc;
    if (p->bk > 3 || p->bv > 4) return set_error(BGTQ_ERR_UNSUPPORTED, "chunked prefill supports bK <= 3 and v_bits <= 4");
    cudaError_t e = launch_quantize_append(*p, (cudaStream_t)stream, k, v, batch, t, pos_start, *c, status);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "chunk append launch: %s", cudaGetErrorString(e));
    e = launch_prefill_chunk(*p, (cudaStream_t)stream, q, k, v, batch, t, pos_start, max_prefix, *c, out, out_dtype,
                             scale, ws, status);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "chunk attention launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}

int bgtq_logit_mae(const bgtq_plan* p, void* stream, const void* q, const void* k, const bgtq_cache* c, int64_t t,
                   int batch, float scale, float* mae) {
    int rc = check_plan(p);
    if (rc) return rc;
    if ((rc = check_cache(p, c))) return rc;
    if (batch < 0 || t < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and t must be >= 0");
    if (t > c->capacity) return set_error(BGTQ_ERR_INVALID_ARG, "t exceeds the cache capacity");
    if (batch == 0) return BGTQ_OK;
    if (!q || !k || !mae) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (reinterpret_cast<uintptr_t>(k) & 7) return set_error(BGTQ_ERR_INVALID_ARG, "k must be 8-byte aligned");
    if (p->G > 8) return set_error(BGTQ_ERR_UNSUPPORTED, "at most 8 query heads per KV head");
    if (!(scale > 0.0f) || !std::isfinite(scale)) return set_error(BGTQ_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (t == 0) {
        cudaError_t e = cudaMemsetAsync(mae, 0, sizeof(float) * (size_t)batch * p->H * p->G, (cudaStream_t)stream);
        if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "logit_mae: %s", cudaGetErrorString(e));
        return BGTQ_OK;
    }
    cudaError_t e = launch_logit_mae(*p, (cudaStream_t)stream, q, k, *c, t, batch, scale, mae);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "logit_mae launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}

int bgtq_dequant_debug(const bgtq_plan* p, void* stream, const bgtq_cache* c, int batch, int b, int head, int64_t t0,
                       int64_t t1, float* k_out, float* v_out, int codec_domain) {
    int rc = check_plan(p);
    if (rc) return rc;
    if ((rc = check_cache(p, c))) return rc;
    if (b < 0 || b >= batch || head < 0 || head >= p->H) return set_error(BGTQ_ERR_INVALID_ARG, "b/head out of range");
    if (t0 < 0 || t1 < t0 || t1 > c->capacity) return set_error(BGTQ_ERR_INVALID_ARG, "token range outside the capacity");
    if (t1 == t0 || (!k_out && !v_out)) return BGTQ_OK;
    cudaError_t e = launch_dequant(*p, (cudaStream_t)stream, *c, batch, b, head, t0, t1, k_out, v_out, codec_domain);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "dequant launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}

}  // extern "C"
