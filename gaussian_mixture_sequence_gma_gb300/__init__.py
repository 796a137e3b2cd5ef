"""GB300-native forward pass of Gaussian Mixture Attention (GMA).

Importing the package loads nothing native; ``gaussian_mixture_sequence_gma_gb300.gma``
loads ``libgma.so`` on first use and raises if it has not been built.
"""
__version__ = "0.1.0"
