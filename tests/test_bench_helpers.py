"""Host-side bookkeeping of bench.py: the algorithmic bytes of the insert and
sparse steps and the size of the insert step.  CPU only."""
import bench
from oracle import sparse as OS
from paged_attention_quantized_gb300 import workloads as W


def test_insert_step_writes_16384_new_tokens_for_every_recipe():
    for name in ("bf16", "e4m3", "int8", "int4", "latent"):
        B = W._SHAPES[name][0]
        assert B * bench.INSERT_NEW_TOKENS[name] == 16384, name


def test_insert_bytes():
    w = W.make("int8", B=3, L_lo=300, L_hi=400, n=5)
    rows = 3 * 5 * w.Hkv
    # f16 rows in (2 bytes per value), one code byte per value out, K and V
    assert bench.insert_bytes(w) == 2 * rows * (128 * 2 + 128)
    w = W.make("int4", B=3, L_lo=300, L_hi=400, n=5)
    assert bench.insert_bytes(w) == 2 * rows * (128 * 2 + 64)
    w = W.make("latent", B=2, L_lo=300, L_hi=400, Hq=16, n=3)
    # one plane: 576 bf16 values in, 576 E4M3 codes and one fp32 scale out
    assert bench.insert_bytes(w) == 2 * 3 * (576 * 2 + 576 + 4)


def test_selected_counts_match_the_oracle_sets():
    w = W.make("qsa", B=2, L_lo=200, L_hi=300, n=7)
    sel = W.make_selection(w, k=50, seed=1)
    got = bench.selected_counts(w, sel)
    L = w.context_lens.tolist()
    want = [OS.selected(sel[b, j].numpy(), L[b] - (w.n - 1 - j)).size for b in range(2) for j in range(7)]
    assert got == want and all(0 < c <= 50 for c in got)


def test_default_run_covers_every_configuration_largest_last():
    # one line per benchmark configuration; the last (the headline) is the
    # largest in tokens and in work: the single-latent MQA batch
    assert set(bench.ALL_CONFIGS) == set(W.CONFIG_NAMES)
    assert bench.ALL_CONFIGS[-1] == "latent"
