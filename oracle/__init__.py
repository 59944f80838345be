"""CPU oracle for FP8 (E4M3 / E5M2) KV-cache quantization and attention over the
paged cache: plain, slow, float64 numpy, written from the pages' statement
of the method.

This package is TEST INFRASTRUCTURE.  Only the tests, the smoke check and
the bench's CPU-baseline leg may import it; the library's product path never
does, and the two share no code.

Modules
-------
e4m3       the E4M3 codec (decode table from the format fields; saturating
           round-to-nearest-even encode; quantize = encode(fl32(x / s))).
e5m2       the E5M2 codec, written the same way.
kv_cache   the paged cache write (K pages [P][D], V pages [D][P]) with
           per-head or per-token dynamic scales, query quantization, the KV
           byte formulas.
attention  paged decode (full / sliding window, FP8 / BF16 cache), the
           log-sum-exp merge of partial results, chunked causal prefill,
           and a planted-defect variant (reduced accumulator) used only to
           show the long-context test is sensitive.

Pins (tests/test_oracle_*.py)
-----------------------------
codec       worked examples of "FP8 and KV cache" (tests/golden), the format's
            closed forms, torch's float8_e4m3fn cast on a dense bit sample and
            on every tie, brute force over all codes, round-trip invariant;
            E5M2: numpy's float16 (its top byte), integer rounding of every
            float16, torch's float8_e5m2, brute force.
per-token   the page's per-token example (scales 3.2/448 and 180/448 found
            from the tokens), reduction to the per-head path, brute force.
cache       per-element brute force, sentinel bytes, skipped / bad slots,
            identity vs permuted block tables.
bytes       every byte count and time the pages print for the formula.
attention   pure-Python brute force, closed forms (constant V, zero K, one
            token, needle), split / merge, page permutation, window, the last
            prefill row vs decode, sensitivity to a 14-bit accumulator.

Prefill P8: the "final" mode (P8 against the row's final maximum) is pinned
by brute force; the "mirror" mode's tile loop is pinned against the
single-pass formula (equal without P rounding for any tile size, equal with
it when the row maximum sits in the first tile).  Which E4M3 code a float32
exponential near a rounding midpoint gets is not pinned bit for bit (the
tolerance covers one step).
"""
