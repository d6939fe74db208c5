"""Rotation ablation through the GPU path: rotated INT2 beats naive INT2.

With four outlier channels per head (x20), quantising keys in their own basis
lets the outliers set every token-group's scale; a rotation spreads them.  Both
the Hadamard-only rotation and OSCAR's must cut the logit error and the
attention KL well below naive INT2 on the same seeded layer.  Which of the two
rotations is better depends on the query statistics: on that law (axis-aligned
outliers, full-rank query covariance) the Hadamard rotation alone already gives
every channel equal query importance.  On the shared-subspace law -- queries with
four dominant directions that the keys share -- the query eigenbasis must cut the
logit error below the Hadamard-only rotation's.
"""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_rotations_beat_naive_int2():
    from bit_rotated_kv_decode_gb300 import ablation, build
    build.build()
    r = ablation.run(tokens=2048 + 320, queries=2, clip=0.9)["results"]
    for variant in ("hadamard", "oscar"):
        assert r[variant]["logit_rel"] < 0.6 * r["naive"]["logit_rel"], r
        assert r[variant]["kl"] < 0.6 * r["naive"]["kl"], r


def test_rotations_beat_naive_int2_at_group64():
    # two {s, z} per token-head: the cache's 5120-byte records are read back per group
    from bit_rotated_kv_decode_gb300 import ablation, build
    build.build()
    r = ablation.run(tokens=2048 + 320, queries=2, clip=0.9, group=64)["results"]
    for variant in ("hadamard", "oscar"):
        assert r[variant]["logit_rel"] < 0.6 * r["naive"]["logit_rel"], r
        assert r[variant]["kl"] < 0.6 * r["naive"]["kl"], r
    # finer groups: the output error is no worse than half again the 128-group one
    r128 = ablation.run(tokens=2048 + 320, queries=2, clip=0.9)["results"]
    assert r["oscar"]["logit_rel"] < 1.5 * r128["oscar"]["logit_rel"], (r, r128)


@pytest.mark.parametrize("group", [128, 64])
def test_query_eigenbasis_beats_hadamard_on_shared_subspace(group):
    from bit_rotated_kv_decode_gb300 import ablation, build
    build.build()
    r = ablation.run(tokens=2048 + 320, queries=4, clip=0.9, group=group, law="subspace",
                     variants=("naive", "hadamard", "oscar"))["results"]
    assert r["hadamard"]["logit_rel"] < r["naive"]["logit_rel"], r
    assert r["oscar"]["logit_rel"] < 0.95 * r["hadamard"]["logit_rel"], r

