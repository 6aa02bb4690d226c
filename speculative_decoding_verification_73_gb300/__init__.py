"""GB300-native batched draft-verify step of speculative decoding.

``binding`` wraps the C-ABI library ``libspecverify.so`` (built from
``csrc/`` by ``build.py``); ``workloads`` builds seeded synthetic inputs.
"""
