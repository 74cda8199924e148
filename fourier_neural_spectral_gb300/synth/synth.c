/* synth.c -- seeded synthetic inputs shared by the tests, the benchmark and the
 * oracle checks.  Holds no arithmetic of the spectral layer itself: only a
 * counter-based random generator and the recipes that turn its draws into x and w.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014).  Stream (seed, s) starts from state
 *   key = mix64(mix64(seed) + s)
 * and draw j (j = 0, 1, ...) is mix64(key + (j + 1) * 0x9E3779B97F4A7C15), i.e.
 * the j-th output of splitmix64's next() from that state.  Because each draw is a
 * pure function of (seed, s, j), any slice can be produced independently and in
 * parallel with identical bytes.
 *
 *   uniform(j) = (draw(j) >> 11) * 2^-53                      in [0, 1)
 *   normal(j)  = sqrt(-2 ln(1 - uniform(2j))) * cos(2 pi uniform(2j + 1))
 *                (Box-Muller, one output per pair of draws, double precision)
 *
 * Values are computed in double and rounded once to float32.
 */
#include <math.h>
#include <stdint.h>

static const double kTwoPi = 6.283185307179586476925286766559005768;
#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed) + stream);
}

static inline double uniform_at(uint64_t key, uint64_t j) {
    return (double)(mix64(key + (j + 1) * GOLDEN) >> 11) * 0x1.0p-53;
}

static inline double normal_at(uint64_t key, uint64_t j) {
    double u1 = 1.0 - uniform_at(key, 2 * j);
    double u2 = uniform_at(key, 2 * j + 1);
    return sqrt(-2.0 * log(u1)) * cos(kTwoPi * u2);
}

uint64_t synth_draw(uint64_t seed, uint64_t stream, uint64_t j) {
    return mix64(stream_key(seed, stream) + (j + 1) * GOLDEN);
}

double synth_uniform(uint64_t seed, uint64_t stream, uint64_t j) {
    return uniform_at(stream_key(seed, stream), j);
}

double synth_normal(uint64_t seed, uint64_t stream, uint64_t j) {
    return normal_at(stream_key(seed, stream), j);
}

/* out[t] = (float) normal(offset + t), t in [0, n) */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, float* out) {
    const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) out[t] = (float)normal_at(key, offset + (uint64_t)t);
}

/* out[t] = (float) (uniform(offset + t) * scale), t in [0, n) */
void synth_uniform_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double scale,
                       float* out) {
    const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) out[t] = (float)(uniform_at(key, offset + (uint64_t)t) * scale);
}

/* "Smooth-ish" planes: per plane pl = b*C + c,
 *   x[h][w] = sum_{j<8} a_j cos(2 pi (p_j h / H + q_j w / W) + phi_j) + 0.1 * n(h, w)
 * with p_j, q_j uniform integers in [-4, 4], a_j ~ N(0, 1/4), phi_j ~ U[0, 2 pi),
 * all drawn from stream 3 at counters (pl * 8 + j) * 5 + {0..4}, and the noise
 * n ~ N(0, 1) from stream 1 at the element's flat index. */
void synth_smooth_f32(uint64_t seed, int B, int C, int H, int W, float* out) {
    const uint64_t kp = stream_key(seed, 3);
    const uint64_t kn = stream_key(seed, 1);
    const int64_t planes = (int64_t)B * C;
    const int64_t hw = (int64_t)H * W;
#pragma omp parallel for schedule(static)
    for (int64_t pl = 0; pl < planes; ++pl) {
        int p[8], q[8];
        double a[8], ph[8];
        for (int j = 0; j < 8; ++j) {
            uint64_t c0 = ((uint64_t)pl * 8 + j) * 5;
            p[j] = (int)floor(uniform_at(kp, c0) * 9.0) - 4;
            q[j] = (int)floor(uniform_at(kp, c0 + 1) * 9.0) - 4;
            double u1 = 1.0 - uniform_at(kp, c0 + 2), u2 = uniform_at(kp, c0 + 3);
            a[j] = 0.5 * sqrt(-2.0 * log(u1)) * cos(kTwoPi * u2);
            ph[j] = kTwoPi * uniform_at(kp, c0 + 4);
        }
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t w = 0; w < W; ++w) {
                double v = 0.0;
                for (int j = 0; j < 8; ++j) {
                    /* phase numerator p*h*W + q*w*H reduced modulo H*W */
                    int64_t num = ((int64_t)p[j] * h * W + (int64_t)q[j] * w * H) % hw;
                    if (num < 0) num += hw;
                    v += a[j] * cos(kTwoPi * (double)num / (double)hw + ph[j]);
                }
                int64_t flat = pl * hw + h * W + w;
                v += 0.1 * normal_at(kn, (uint64_t)flat);
                out[flat] = (float)v;
            }
        }
    }
}
