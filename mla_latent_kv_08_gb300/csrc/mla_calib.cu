// Calibration of the rotated-INT2 cache, the library's own: the per-layer covariance
// Sigma = X^T X of calibration latents (GPU, fp64), its eigenbasis in ascending
// eigenvalue order with a sign rule (host), the up-projection-aware variant (the
// eigenbasis of S^1/2 M S^1/2 with M the projection energy of W_UK and W_UV), and
// the per-group clip thresholds, the pct-th percentile of |X . R| (GPU projection,
// host selection).
//   Source: "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10),
//   maintainer reply, "How the rotation adapts to the latent" (Sigma = c^T c, eigh in
//   ascending order so that low-variance directions share INT2 groups, clip
//   thresholds fit on the rotated latent), and the "open refinement" paragraph after
//   it (weighting the latent directions by what the up-projection does with them).
//
// The symmetric eigensolver is Householder tridiagonalisation followed by the
// implicit symmetric QL iteration with Wilkinson shifts (Golub & Van Loan, Matrix
// Computations, sections 8.3.1 and 8.3.3), written here from that description.
#include "mla_internal.cuh"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

namespace mla {
namespace calib {

// ---------------------------------------------------------------- GPU: Gram matrices
// G[i][j] (+)= sum_t x(t, i) x(t, j) in fp64 for a [T, d] operand read through one
// of two layouts: rows (x(t, i) = X[t * d + i]) or the transposed heads of a
// [H, d, m] tensor (t = h * m + v, x(t, i) = X[(h * d + i) * m + v]). A CTA owns a
// 64 x 64 tile of G and runs over all T rows (no atomics: deterministic); each
// thread owns a 4 x 4 block.
enum { kRows = 0, kHeadsT = 1 };

template <typename T> __device__ __forceinline__ double to_f64(T v);
template <> __device__ __forceinline__ double to_f64<double>(double v) { return v; }
template <> __device__ __forceinline__ double to_f64<float>(float v) { return (double)v; }
template <> __device__ __forceinline__ double to_f64<__nv_bfloat16>(__nv_bfloat16 v) { return (double)__bfloat162float(v); }

template <typename T, int LAYOUT>
__global__ void __launch_bounds__(256) gram_kernel(const T *X, long long nT, int d, int m, double *G, int accumulate) {
    __shared__ double sa[16][64 + 1];
    __shared__ double sb[16][64 + 1];
    const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    double acc[4][4] = {};
    auto at = [&](long long t, int i) -> double {
        if (LAYOUT == kRows) return to_f64(X[t * d + i]);
        const long long h = t / m, v = t % m;
        return to_f64(X[(h * d + i) * m + v]);
    };
    for (long long t0 = 0; t0 < nT; t0 += 16) {
        for (int e = threadIdx.x; e < 16 * 64; e += 256) {
            const int tt = e >> 6, c = e & 63;
            const long long t = t0 + tt;
            sa[tt][c] = (t < nT && i0 + c < d) ? at(t, i0 + c) : 0.0;
            sb[tt][c] = (t < nT && j0 + c < d) ? at(t, j0 + c) : 0.0;
        }
        __syncthreads();
#pragma unroll 4
        for (int tt = 0; tt < 16; ++tt) {
            double a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = sa[tt][4 * ty + u];
                b[u] = sb[tt][4 * tx + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fma(a[u], b[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = i0 + 4 * ty + u;
        if (i >= d) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int j = j0 + 4 * tx + v;
            if (j >= d) continue;
            double *g = G + (size_t)i * d + j;
            *g = accumulate ? *g + acc[u][v] : acc[u][v];
        }
    }
}

template <int LAYOUT>
static cudaError_t launch_gram(const void *X, int dtype, long long nT, int d, int m, double *G, int accumulate,
                               cudaStream_t st) {
    dim3 grid((d + 63) / 64, (d + 63) / 64);
    switch (dtype) {
        case MLA_DTYPE_F64: gram_kernel<double, LAYOUT><<<grid, 256, 0, st>>>((const double *)X, nT, d, m, G, accumulate); break;
        case MLA_DTYPE_F32: gram_kernel<float, LAYOUT><<<grid, 256, 0, st>>>((const float *)X, nT, d, m, G, accumulate); break;
        default:
            gram_kernel<__nv_bfloat16, LAYOUT><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)X, nT, d, m, G, accumulate);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- GPU: |X . R|
// absY[t][j] = |sum_k x(t, k) R[k][j]|, fp64; a CTA computes a 64 x 64 tile.
template <typename T>
__global__ void __launch_bounds__(256) project_abs_kernel(const T *X, long long n, int d, const double *R, double *absY) {
    __shared__ double sx[64][16 + 1];
    __shared__ double sr[16][64 + 1];
    const long long t0 = (long long)blockIdx.y * 64;
    const int j0 = blockIdx.x * 64;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    double acc[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += 16) {
        for (int e = threadIdx.x; e < 64 * 16; e += 256) {
            const int rr = e >> 4, kk = e & 15;
            const long long t = t0 + rr;
            sx[rr][kk] = (t < n && k0 + kk < d) ? to_f64(X[t * d + k0 + kk]) : 0.0;
            const int kr = e >> 6, c = e & 63;
            sr[kr][c] = (k0 + kr < d && j0 + c < d) ? R[(size_t)(k0 + kr) * d + j0 + c] : 0.0;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < 16; ++kk) {
            double a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = sx[4 * ty + u][kk];
                b[u] = sr[kk][4 * tx + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fma(a[u], b[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const long long t = t0 + 4 * ty + u;
        if (t >= n) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int j = j0 + 4 * tx + v;
            if (j < d) absY[t * d + j] = fabs(acc[u][v]);
        }
    }
}

// ---------------------------------------------------------------- host: eigensolver
// Symmetric A [n x n] (row-major, overwritten) -> eigenvalues w (unsorted) and
// eigenvectors as the ROWS of ZT [n x n] (row c is the eigenvector of w[c]; kept
// transposed so that the rotations below touch contiguous rows). Returns false if
// the iteration does not converge.
static bool symmetric_eigen(std::vector<double> &A, int n, std::vector<double> &w, std::vector<double> &ZT) {
    // 1. Householder tridiagonalisation: Q^T A Q = T; ZT accumulates Q^T.
    std::vector<double> diag(n), off(n, 0.0);
    ZT.assign((size_t)n * n, 0.0);
    for (int i = 0; i < n; ++i) ZT[(size_t)i * n + i] = 1.0;
    std::vector<double> v(n), p(n), q(n), t(n);
    for (int k = 0; k + 2 < n; ++k) {
        // x = A[k+1:, k]; reflector H = I - beta v v^T with H x = alpha e_1
        double sigma = 0.0;
        for (int i = k + 1; i < n; ++i) sigma += A[(size_t)i * n + k] * A[(size_t)i * n + k];
        const double x0 = A[(size_t)(k + 1) * n + k];
        const double nx = std::sqrt(sigma);
        if (nx == 0.0) continue;                    // column already reduced
        const double alpha = x0 > 0.0 ? -nx : nx;  // avoids cancellation in v_0
        for (int i = k + 1; i < n; ++i) v[i] = A[(size_t)i * n + k];
        v[k + 1] = x0 - alpha;
        double vv = 0.0;
        for (int i = k + 1; i < n; ++i) vv += v[i] * v[i];
        if (vv == 0.0) continue;
        const double beta = 2.0 / vv;
        // trailing block A <- H A H: p = beta A v, q = p - (beta p.v / 2) v,
        // A -= v q^T + q v^T
        for (int i = k + 1; i < n; ++i) {
            double s = 0.0;
            const double *Ai = &A[(size_t)i * n];
            for (int j = k + 1; j < n; ++j) s += Ai[j] * v[j];
            p[i] = beta * s;
        }
        double pv = 0.0;
        for (int i = k + 1; i < n; ++i) pv += p[i] * v[i];
        const double c = 0.5 * beta * pv;
        for (int i = k + 1; i < n; ++i) q[i] = p[i] - c * v[i];
        for (int i = k + 1; i < n; ++i) {
            double *Ai = &A[(size_t)i * n];
            for (int j = k + 1; j < n; ++j) Ai[j] -= v[i] * q[j] + q[i] * v[j];
        }
        for (int i = k + 2; i < n; ++i) {
            A[(size_t)i * n + k] = 0.0;
            A[(size_t)k * n + i] = 0.0;
        }
        A[(size_t)(k + 1) * n + k] = alpha;
        A[(size_t)k * n + k + 1] = alpha;
        // Q <- Q H, i.e. ZT <- H ZT on rows k+1..n-1: ZT -= beta v (v^T ZT)
        std::fill(t.begin(), t.end(), 0.0);
        for (int j = k + 1; j < n; ++j) {
            const double vj = v[j];
            const double *Zj = &ZT[(size_t)j * n];
            for (int r = 0; r < n; ++r) t[r] += vj * Zj[r];
        }
        for (int j = k + 1; j < n; ++j) {
            const double bv = beta * v[j];
            double *Zj = &ZT[(size_t)j * n];
            for (int r = 0; r < n; ++r) Zj[r] -= bv * t[r];
        }
    }
    for (int i = 0; i < n; ++i) diag[i] = A[(size_t)i * n + i];
    for (int i = 0; i + 1 < n; ++i) off[i] = A[(size_t)(i + 1) * n + i];
    off[n - 1] = 0.0;
    // 2. Implicit QL with Wilkinson shifts on (diag, off); off[i] couples rows i and
    //    i + 1. Each plane rotation of rows i, i+1 of T is applied to rows i, i+1 of ZT.
    for (int l = 0; l < n; ++l) {
        int iter = 0;
        for (;;) {
            int m = l;
            for (; m + 1 < n; ++m) {
                const double dd = std::fabs(diag[m]) + std::fabs(diag[m + 1]);
                if (std::fabs(off[m]) <= 1e-300 + 2.2e-16 * dd) break;
            }
            if (m == l) break;                      // diag[l] has converged
            if (++iter > 60) return false;
            // shift: the eigenvalue of the leading 2 x 2 block closer to diag[l]
            double g = (diag[l + 1] - diag[l]) / (2.0 * off[l]);
            double r = std::hypot(g, 1.0);
            g = diag[m] - diag[l] + off[l] / (g + (g >= 0.0 ? r : -r));
            double s = 1.0, c = 1.0, shift_acc = 0.0;
            bool split = false;
            for (int i = m - 1; i >= l; --i) {
                double f = s * off[i];
                const double b = c * off[i];
                r = std::hypot(f, g);
                off[i + 1] = r;
                if (r == 0.0) {                      // the block splits: restart on it
                    diag[i + 1] -= shift_acc;
                    off[m] = 0.0;
                    split = true;
                    break;
                }
                s = f / r;
                c = g / r;
                g = diag[i + 1] - shift_acc;
                r = (diag[i] - g) * s + 2.0 * c * b;
                shift_acc = s * r;
                diag[i + 1] = g + shift_acc;
                g = c * r - b;
                double *Zi = &ZT[(size_t)i * n], *Zi1 = &ZT[(size_t)(i + 1) * n];
                for (int k = 0; k < n; ++k) {
                    f = Zi1[k];
                    Zi1[k] = s * Zi[k] + c * f;
                    Zi[k] = c * Zi[k] - s * f;
                }
            }
            if (split) continue;
            diag[l] -= shift_acc;
            off[l] = g;
            off[m] = 0.0;
        }
    }
    w = diag;
    return true;
}

// Ascending order of w (stable), then each column flipped so that its largest-
// magnitude entry (the first one on ties) is positive. R64 / R32 optional.
static void sort_and_sign(const std::vector<double> &w, const std::vector<double> &ZT, int n, double *eigvals,
                          double *R64, float *R32) {
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return w[a] < w[b]; });
    for (int c = 0; c < n; ++c) {
        const int src = order[c];
        if (eigvals) eigvals[c] = w[src];
        int arg = 0;
        double best = -1.0;
        for (int r = 0; r < n; ++r) {
            const double a = std::fabs(ZT[(size_t)src * n + r]);
            if (a > best) { best = a; arg = r; }
        }
        const double sgn = ZT[(size_t)src * n + arg] < 0.0 ? -1.0 : 1.0;
        for (int r = 0; r < n; ++r) {
            const double val = sgn * ZT[(size_t)src * n + r];
            if (R64) R64[(size_t)r * n + c] = val;
            if (R32) R32[(size_t)r * n + c] = (float)val;
        }
    }
}

}  // namespace calib
}  // namespace mla

using namespace mla;

extern "C" {

mla_status mla_calib_covariance(const void *X, int64_t n, int32_t d, int32_t dtype, double *sigma, void *stream) {
    if (!X || !sigma || n < 1 || d < 1 || d > 4096 || dtype < MLA_DTYPE_F64 || dtype > MLA_DTYPE_BF16)
        return MLA_ERR_INVALID;
    return calib::launch_gram<calib::kRows>(X, dtype, n, d, 0, sigma, 0, (cudaStream_t)stream) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}

mla_status mla_calib_projection_energy(const void *W_UK, const void *W_UV, int32_t H, int32_t d_n, int32_t r,
                                       int32_t d_v, int32_t dtype, double *M, void *stream) {
    if (!W_UK || !W_UV || !M || H < 1 || d_n < 1 || r < 1 || r > 4096 || d_v < 1 || dtype < MLA_DTYPE_F64 ||
        dtype > MLA_DTYPE_BF16)
        return MLA_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    // sum_h W_UK[h]^T W_UK[h]: the Gram matrix of the H * d_n rows of W_UK
    if (calib::launch_gram<calib::kRows>(W_UK, dtype, (long long)H * d_n, r, 0, M, 0, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    // + sum_h W_UV[h] W_UV[h]^T: the Gram matrix of the H * d_v columns of W_UV
    if (calib::launch_gram<calib::kHeadsT>(W_UV, dtype, (long long)H * d_v, r, d_v, M, 1, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_OK;
}

mla_status mla_calib_project_abs(const void *X, int64_t n, int32_t d, int32_t dtype, const double *R, double *absY,
                                 void *stream) {
    if (!X || !R || !absY || n < 1 || d < 1 || d > 4096 || dtype < MLA_DTYPE_F64 || dtype > MLA_DTYPE_BF16)
        return MLA_ERR_INVALID;
    dim3 grid((d + 63) / 64, (unsigned)((n + 63) / 64));
    cudaStream_t st = (cudaStream_t)stream;
    switch (dtype) {
        case MLA_DTYPE_F64: calib::project_abs_kernel<double><<<grid, 256, 0, st>>>((const double *)X, n, d, R, absY); break;
        case MLA_DTYPE_F32: calib::project_abs_kernel<float><<<grid, 256, 0, st>>>((const float *)X, n, d, R, absY); break;
        default: calib::project_abs_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)X, n, d, R, absY);
    }
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status mla_calib_eigh(const double *A, int32_t d, double *eigvals, double *R64, float *R32) {
    if (!A || d < 1 || d > 4096 || (!eigvals && !R64 && !R32)) return MLA_ERR_INVALID;
    std::vector<double> M(A, A + (size_t)d * d), w, ZT;
    for (int i = 0; i < d; ++i)                     // symmetrise (the lower triangle wins)
        for (int j = i + 1; j < d; ++j) M[(size_t)i * d + j] = M[(size_t)j * d + i];
    if (!calib::symmetric_eigen(M, d, w, ZT)) return MLA_ERR_UNSUPPORTED;
    calib::sort_and_sign(w, ZT, d, eigvals, R64, R32);
    return MLA_OK;
}

mla_status mla_calib_eigh_weighted(const double *S, const double *M, int32_t d, double *eigvals, double *R64,
                                   float *R32) {
    if (!S || !M || d < 1 || d > 4096 || (!eigvals && !R64 && !R32)) return MLA_ERR_INVALID;
    const size_t dd = (size_t)d * d;
    // S^1/2 = V diag(sqrt(max(w, 0))) V^T from the eigenbasis of S
    std::vector<double> Sc(S, S + dd), w, VT;
    for (int i = 0; i < d; ++i)
        for (int j = i + 1; j < d; ++j) Sc[(size_t)i * d + j] = Sc[(size_t)j * d + i];
    if (!calib::symmetric_eigen(Sc, d, w, VT)) return MLA_ERR_UNSUPPORTED;
    std::vector<double> Sh(dd, 0.0), T(dd, 0.0), G(dd, 0.0);
    // Sh = sum_k sqrt(w_k) v_k v_k^T (v_k = row k of VT)
    for (int k = 0; k < d; ++k) {
        const double sk = std::sqrt(std::max(w[k], 0.0));
        if (sk == 0.0) continue;
        const double *vk = &VT[(size_t)k * d];
        for (int i = 0; i < d; ++i) {
            const double a = sk * vk[i];
            if (a == 0.0) continue;
            double *Si = &Sh[(size_t)i * d];
            for (int j = 0; j < d; ++j) Si[j] += a * vk[j];
        }
    }
    // G = S^1/2 M S^1/2, symmetrised
    for (int i = 0; i < d; ++i)
        for (int k = 0; k < d; ++k) {
            const double a = Sh[(size_t)i * d + k];
            if (a == 0.0) continue;
            for (int j = 0; j < d; ++j) T[(size_t)i * d + j] += a * M[(size_t)k * d + j];
        }
    for (int i = 0; i < d; ++i)
        for (int k = 0; k < d; ++k) {
            const double a = T[(size_t)i * d + k];
            if (a == 0.0) continue;
            for (int j = 0; j < d; ++j) G[(size_t)i * d + j] += a * Sh[(size_t)k * d + j];
        }
    for (int i = 0; i < d; ++i)
        for (int j = i + 1; j < d; ++j) {
            const double a = 0.5 * (G[(size_t)i * d + j] + G[(size_t)j * d + i]);
            G[(size_t)i * d + j] = G[(size_t)j * d + i] = a;
        }
    std::vector<double> wg, ZT;
    if (!calib::symmetric_eigen(G, d, wg, ZT)) return MLA_ERR_UNSUPPORTED;
    calib::sort_and_sign(wg, ZT, d, eigvals, R64, R32);
    return MLA_OK;
}

mla_status mla_calib_thresholds(double *absY, int64_t n, int32_t d, int32_t group_size, double pct, float *clip) {
    if (!absY || !clip || n < 1 || d < 1 || group_size < 1 || d % group_size || !(pct >= 0.0 && pct <= 100.0))
        return MLA_ERR_INVALID;
    const int ng = d / group_size;
    const long long N = (long long)n * group_size;
    std::vector<double> vals((size_t)N);
    // linear interpolation between the order statistics around (N - 1) * pct / 100
    const double pos = (double)(N - 1) * (pct / 100.0);
    const long long lo = (long long)std::floor(pos);
    const double frac = pos - (double)lo;
    for (int g = 0; g < ng; ++g) {
        size_t k = 0;
        for (long long t = 0; t < n; ++t)
            for (int j = 0; j < group_size; ++j) vals[k++] = absY[(size_t)t * d + (size_t)g * group_size + j];
        std::nth_element(vals.begin(), vals.begin() + lo, vals.end());
        const double a = vals[(size_t)lo];
        double b = a;
        if (lo + 1 < N) b = *std::min_element(vals.begin() + lo + 1, vals.end());
        const double v = frac < 0.5 ? a + (b - a) * frac : b - (b - a) * (1.0 - frac);
        clip[g] = (float)v;
    }
    return MLA_OK;
}

}  // extern "C"
