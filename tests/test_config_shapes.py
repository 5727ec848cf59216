"""The generator's large configs carry the shapes the pages print (CPU)."""
import os

from mixture_experts_layer_router_gb300.synth import CONFIGS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layer_shapes.txt")


def _load():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = (s.strip() for s in line.split("="))
        vals[key] = int(val)
    return vals


def test_mai_base_1_shape():
    g = _load()
    c = CONFIGS["mai-base-1"]
    assert (c.d, c.l, c.E, c.k, c.F, c.Fs) == (
        g["mai_base_1.hidden"], g["mai_base_1.latent"], g["mai_base_1.experts"],
        g["mai_base_1.top_k"], g["mai_base_1.expert_ffn"], 0)
    assert c.l == 512 * g["mai_base_1.latent_div_512"]
    # ladder rule from the MAI-Base-2 page: hidden = (256/3) * layers, exact
    assert 256 * g["mai_base_1.layers"] == 3 * c.d


def test_mai_base_2_shape():
    g = _load()
    c = CONFIGS["mai-base-2"]
    assert (c.d, c.l, c.k) == (g["mai_base_2.hidden"], g["mai_base_2.latent"], g["mai_base_2.top_k"])
    assert 256 * g["mai_base_2.layers"] == 3 * c.d
    # one GPU holds 256 of the pages' 512 experts; the shared expert is present
    assert c.E == g["mai_base_2.experts"] // 2 and c.Fs > 0


def test_small_configs_are_multiples_of_128():
    for c in CONFIGS.values():
        for v in (c.d, c.l, c.F):
            assert v % 128 == 0
        assert c.Fs % 128 == 0
