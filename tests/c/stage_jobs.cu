// Host-side check of the staging jobs of ssu_update_from_host (no GPU needed): for many
// operand geometries, expanding a job vector by vector with the kernel's own address
// arithmetic must copy exactly the bytes of the original rows, each once, into the dense
// destination order, with every vector aligned to its width.  Prints "ok" or the first
// failing geometry.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "ssu_stage.cuh"

static unsigned long long rng_state = 0x9E3779B97F4A7C15ull;
static long long draw(long long n) {  // splitmix64, uniform in [0, n)
    unsigned long long z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return static_cast<long long>(z % static_cast<unsigned long long>(n));
}

int main() {
    const long long elems[] = {1, 2, 4, 8};
    for (int trial = 0; trial < 20000; ++trial) {
        const long long esz = elems[draw(4)];
        const long long outer = 1 + draw(6), inner = 1 + draw(5);
        const long long row_elems = 1 + draw(40);
        const long long row_bytes = row_elems * esz;
        // inner stride: contiguous, padded, or broadcast; outer stride: contiguous or padded
        long long s_inner_e;
        switch (draw(3)) {
            case 0: s_inner_e = row_elems; break;
            case 1: s_inner_e = row_elems + draw(9); break;
            default: s_inner_e = draw(2) ? 0 : row_elems + 1;
        }
        const long long span_e = (inner - 1) * s_inner_e + row_elems;
        const long long s_outer_e = draw(2) ? span_e : span_e + draw(17);
        const long long base_off = draw(8) * esz;  // source offset within an aligned buffer
        const long long src_bytes = base_off + (outer - 1) * s_outer_e * esz + span_e * esz;
        // a 256-byte aligned base, as the allocator gives, then the operand's own offset
        std::vector<unsigned char> big(static_cast<size_t>(src_bytes + 512));
        unsigned char *abuf = reinterpret_cast<unsigned char *>(
            (reinterpret_cast<unsigned long long>(big.data()) + 255) & ~255ull);
        const unsigned char *s = abuf + base_off;
        long long chunk0 = 17;
        const StageJob J = stage_job(s, nullptr, outer, inner, s_outer_e * esz, s_inner_e * esz,
                                     row_bytes, chunk0);
        const long long dense = outer * inner * row_bytes;
        std::vector<long long> got(static_cast<size_t>(dense), -1);
        const long long vectors = chunk0 - 17;
        bool ok = J.chunk0 == 17 && vectors * J.vec == dense;
        for (long long c = 0; ok && c < vectors; ++c) {
            long long so, dof;
            stage_offsets(J, c, so, dof);
            const unsigned long long a = reinterpret_cast<unsigned long long>(s) + so;
            if (a % J.vec != 0 || dof % J.vec != 0 || dof < 0 || dof + J.vec > dense) ok = false;
            for (int i = 0; ok && i < J.vec; ++i) {
                if (got[dof + i] != -1) ok = false;
                got[dof + i] = so + i;
            }
        }
        // reference: dense row r = (o, i) holds the row at o * s_outer + i * s_inner
        for (long long o = 0; ok && o < outer; ++o)
            for (long long i = 0; ok && i < inner; ++i)
                for (long long e = 0; ok && e < row_bytes; ++e) {
                    const long long d = (o * inner + i) * row_bytes + e;
                    const long long want = o * s_outer_e * esz + i * s_inner_e * esz + e;
                    if (got[d] != want) ok = false;
                }
        if (!ok) {
            printf("FAIL trial %d: esz %lld outer %lld inner %lld row %lld s_outer %lld "
                   "s_inner %lld base %lld -> vec %d inner %lld row_bytes %lld\n",
                   trial, esz, outer, inner, row_elems, s_outer_e, s_inner_e, base_off, J.vec,
                   J.inner, J.row_bytes);
            return 1;
        }
    }
    printf("ok\n");
    return 0;
}
