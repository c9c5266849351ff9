// Host check of the shared-memory plans of the Gated DeltaNet decode step
// kernel: for every ring length and a range of items per CTA, the layout the
// launcher picks fits in 227 KiB, the tensor-core operand regions start on
// 1024-byte boundaries (the 128-byte swizzle atoms), and the fold phase's
// operands (including the 96 rows a Gram MMA reads past the projection
// operand) stay inside its plan.  Prints one line per case and "ok" at the end.
#include <cstdio>

#include "gdn_fold_tc.cuh"

using namespace rssm;

int main() {
    const int my_cases[] = {1, 2, 54, 128, 216, 512, 513, 1024, 4096};
    bool ok = true;
    for (int L = 1; L <= kGdnMaxL; ++L) {
        for (int my : my_cases) {
            // the launcher's choice: the fold phase when it fits, stages from 6 down
            int stages = 0, total = 0;
            bool fold = my <= kFtMaxMy;
            for (int pass = 0; pass < 2 && !stages; ++pass, fold = false) {
                for (int s = 6; s >= 2; --s) {
                    const GStepSmem lay(L, s, 4, my, fold);
                    if (lay.total <= 227 * 1024) { stages = s; total = lay.total; break; }
                }
                if (stages) break;
            }
            const FTSmem f(L);
            const bool aligned = f.planes_off % 1024 == 0 && f.pop_off % 1024 == 0 && f.kt_off % 1024 == 0;
            // a Gram MMA reads 128 rows x 128 bytes (16 KiB) from the second K-block of
            // the second projection operand: it must end inside the fold plan
            const bool gram_in = f.pop_off + 8192 + 4096 + 16384 <= f.total;
            const bool fits = stages > 0 && total <= 227 * 1024;
            const bool want_fold = my <= kFtMaxMy;
            const bool case_ok = fits && aligned && gram_in && (fold == want_fold);
            std::printf("L %2d items/CTA %4d: stages %d fold phase %d smem %d%s\n", L, my, stages, (int)fold, total,
                        case_ok ? "" : "  <-- bad");
            ok = ok && case_ok;
        }
    }
    std::printf(ok ? "ok\n" : "FAILED\n");
    return ok ? 0 : 1;
}
