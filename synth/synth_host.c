/*
 * Host C twin of the seeded input generator (same definition as
 * synth/__init__.py and synth/synth.cu; the three agree bit for bit).  It
 * exists only for speed: full-size layers have ~10^8 elements per matrix.
 * It holds none of the method's arithmetic.
 */
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_host_key(uint64_t seed, uint64_t tid) { return mix64(seed * GAMMA + mix64(tid)); }

static inline float value(uint64_t key, uint64_t n, float scale)
{
    int s = 0;
    for (int k = 0; k < 3; k++) {
        uint64_t r = mix64(key + (3ull * n + (uint64_t)k + 1ull) * GAMMA);
        s += (int)(r & 0xFFFF) + (int)((r >> 16) & 0xFFFF) + (int)((r >> 32) & 0xFFFF) +
             (int)((r >> 48) & 0xFFFF);
    }
    volatile float t = (float)(s - 393210);   /* exact: |t| < 2^24 */
    volatile float v = t * scale;             /* one IEEE fp32 multiply */
    return v;
}

static inline uint16_t to_bf16(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/*
 * Fill out [n_rows, ld] with rows row_ids[0..n_rows) (or 0..n_rows when
 * row_ids is NULL) of the [*, cols] tensor with key `key`; columns >= cols
 * are zero.  dtype 0 f32, 1 f16, 2 bf16 (raw bits).
 */
void synth_host_fill(void *out, int dtype, const int64_t *row_ids, int64_t n_rows, int64_t cols,
                     int64_t ld, uint64_t key, float scale)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_rows; i++) {
        const int64_t row = row_ids ? row_ids[i] : i;
        for (int64_t c = 0; c < ld; c++) {
            float v = c < cols ? value(key, (uint64_t)(row * cols + c), scale) : 0.0f;
            size_t o = (size_t)i * (size_t)ld + (size_t)c;
            if (dtype == 0)
                ((float *)out)[o] = v;
            else if (dtype == 1)
                ((_Float16 *)out)[o] = (_Float16)v;
            else
                ((uint16_t *)out)[o] = to_bf16(v);
        }
    }
}
