"""Workload table: the seeded synthetic MoE-layer problems.

Each entry fixes the layer shape (T tokens, hidden H, expert intermediate I,
E experts, top-k, local expert range [e0, e1)) and the value distributions of
the inputs. Sizes follow the serving write-up "Hosting Qwen on Blackwell":
prefill of a ~6000-token input with top-8 of 128 experts gives
6000*8/128 = 375 tokens per expert ("Prefillers" section), one prefill rank
holds 32 of the 128 experts (TP=4/EP=4, same section), and decode is bound by
streaming the expert weights from HBM ("Decoders" section).

The skewed workloads add a Zipf-like bias 3*ln(1/(e+1)) to each expert's logit.
"skewed" keeps the local range [32, 64) as the workload is stated; with that
bias almost no pair lands there. "skewed_rank0" is the same logits seen by the
rank that owns [0, 32), which is where the heavy load actually goes.
"""

CONFIGS = {
    "tiny": dict(T=64, H=256, I=128, E=16, k=4, e0=0, e1=16,
                 x_std=1.0, logit_std=1.0, w_std=0.05, zipf_bias=False),
    "prefill_ep_rank": dict(T=6000, H=4096, I=1536, E=128, k=8, e0=0, e1=32,
                            x_std=1.0, logit_std=1.0, w_std=0.02, zipf_bias=False),
    "prefill_full": dict(T=16384, H=4096, I=1536, E=128, k=8, e0=0, e1=128,
                         x_std=1.0, logit_std=1.0, w_std=0.02, zipf_bias=False),
    "decode": dict(T=256, H=4096, I=1536, E=128, k=8, e0=0, e1=128,
                   x_std=1.0, logit_std=1.0, w_std=0.02, zipf_bias=False),
    "skewed": dict(T=6000, H=4096, I=1536, E=128, k=8, e0=32, e1=64,
                   x_std=1.0, logit_std=1.0, w_std=0.02, zipf_bias=True),
    "skewed_rank0": dict(T=6000, H=4096, I=1536, E=128, k=8, e0=0, e1=32,
                         x_std=1.0, logit_std=1.0, w_std=0.02, zipf_bias=True),
}

# "MoE GEMM" section: the decode GEMM benchmark activates every expert with a
# single token.  One EP rank of an EP=N deployment holds n = 128/N experts and
# sees T = n tokens, token t routed (top-1) to local expert t.
for _ep in (1, 2, 4, 8, 16, 32):
    _n = 128 // _ep
    CONFIGS[f"one_token_per_expert_ep{_ep}"] = dict(
        T=_n, H=4096, I=1536, E=128, k=1, e0=0, e1=_n, x_std=1.0, logit_std=1.0, w_std=0.02,
        zipf_bias=False, one_token_per_expert=True)

# tensor ids of the generator streams; weights are indexed by GLOBAL expert id so
# that any local range [e0, e1) sees the same bytes as the full tensor
TID_X, TID_LOGITS, TID_W_GATE, TID_W_UP, TID_W_DOWN = 1, 2, 3, 4, 5
TID_AUX = 16  # free-form streams for unit tests (y rows, weights, ...)


def dims_of(cfg):
    """The (T, H, I, E, k, e0, e1) tuple of a config dict."""
    return tuple(cfg[n] for n in ("T", "H", "I", "E", "k", "e0", "e1"))
